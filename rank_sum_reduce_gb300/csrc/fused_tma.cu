// fused_tma.cu -- rank sum + residual add + RMSNorm for many rows, with the
// rank slices streamed into shared memory by TMA bulk copies.
//
// Same operation as fused.cu (P4 "用 Triton + Symmetric Memory 写一个
// AllReduce + RMSNorm 融合算子", "这个算子在算什么"; rank order and single
// rounding from P1 "1stage：kernel 全文与时间线"), organised for HBM
// throughput on GB300 rather than for one row:
//
//  * one persistent CTA per SM takes rows blockIdx.x, blockIdx.x + grid, ...;
//  * a producer thread walks (row, rank) slices -- x_0 .. x_{W-1}, then the
//    residual -- and issues one cp.async.bulk per slice into a ring of
//    shared-memory slots, signalling an mbarrier with the byte count; it runs
//    up to `slots` slices ahead, so loads stay in flight while the consumers
//    reduce, normalise and store;
//  * consumer warps own fixed 16-byte columns of the row: they fold each rank
//    slice into fp32 accumulators in rank order as it lands, add the
//    residual, store ar / residual_out, then meet at an mbarrier for the
//    row's sum of squares (two when a cluster shares the row) and store
//    norm_out.  The weight row stays in
//    registers for the whole kernel.  At W = 8 the last kRegSlices slices of
//    a row skip the ring: the consumers load their own columns of them;
//  * before the PDL wait, each CTA asks L2 for its first row, so that row's
//    HBM latency passes while the previous grid of the stream finishes (only
//    when there is such a grid still running).
//
// Every mbarrier wait is bounded (about one second of %globaltimer); a wait
// that runs out sets bit 0 of *err, stops the CTA's producer, waits (bounded
// again) for the copies it already issued, and returns.
#include "car_device.cuh"
#include "car_launch.h"

namespace car {
namespace {

// Slices per row loaded by the consumers instead of bulk copies (see run_consumers).
constexpr int kRegSlices = 3;
// First-row L2 prefetch in the prologue: slices requested at once, and how
// long the producer warp looks for the dependency wait's return before it
// requests the rest (see the kernel's prologue).
constexpr int kEarlyPrefetch = 2;
constexpr unsigned long long kPrefetchGraceNs = 100;

struct TmaParams {
  RankPtrs in;
  const uint8_t* residual;
  const uint4* weight;
  uint4* residual_out;
  uint4* norm_out;
  uint4* ar_out;       // may be null
  unsigned int* err;   // bounded-wait failure flag (bit 0)
  float eps;
  float cols;
  int64_t rows;
  int row_bytes;       // N * s
  int vec_per_row;
  int slots;           // ring depth
  int tma_slices;      // leading slices of a row that come by bulk copy (the rest by plain loads)
  int consumers;       // consumer threads (multiple of 32)
  int nranks;
  int cluster;         // CTAs sharing a row (1 or 2): each takes 1/cluster of the columns
};

// Wait for the barrier phase with the given parity; false when the CTA is
// aborting or the wait ran past kWaitLimitNs.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1; i < (1u << 30); i++) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && (*abort || globaltimer() - t0 > kWaitLimitNs)) return false;
  }
  return false;
}
// Same, ignoring the abort flag (used while draining on the way out).
__device__ __forceinline__ bool wait_bounded_cluster(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1; i < (1u << 30); i++) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0 && (*abort || globaltimer() - t0 > kWaitLimitNs)) return false;
  }
  return false;
}
__device__ __forceinline__ bool wait_bounded_drain(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1; i < (1u << 30); i++) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return false;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ uint4 lds16(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Producer: one thread walks this CTA's (row, rank) slices in order and keeps
// the ring full.  Returns after every copy it issued has landed.
__device__ __forceinline__ void run_producer(const TmaParams& p, uint8_t* ring, uint64_t* full, uint64_t* empty,
                                             volatile int* s_abort, int S, int slice, int n, uint32_t crank,
                                             int64_t group, int64_t ngroups) {
  int slot = 0;
  uint32_t phase = 0;
  uint64_t issued = 0;
  bool ok = true;
  for (int64_t row = group; row < p.rows && ok; row += ngroups) {
    const int64_t off = row * (int64_t)p.row_bytes + (int64_t)crank * slice;
    for (int q = 0; q < p.tma_slices; q++) {
      // slot reuse: wait until every consumer warp released its previous fill
      if (issued >= (uint64_t)S && !wait_bounded(&empty[slot], phase ^ 1u, s_abort)) {
        ok = false;
        break;
      }
      const uint8_t* src = (q < n ? static_cast<const uint8_t*>(p.in.p[q]) : p.residual) + off;
      mbar_arrive_expect_tx(&full[slot], (uint32_t)slice);
      bulk_load(ring + (size_t)slot * slice, src, (uint32_t)slice, &full[slot]);
      issued++;
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok) {
    atomicOr(p.err, 1u);
    *s_abort = 1;
  }
  // Make sure no copy is still writing into shared memory: wait (bounded) for
  // the latest fill of every slot that was used.  Copy number c went to slot
  // c % S as that slot's use c / S, which completes the full barrier's phase
  // of parity (c / S) & 1.
  const int used = issued < (uint64_t)S ? (int)issued : S;
  for (int k = 0; k < used; k++) {
    const uint64_t c = issued - 1 - (uint64_t)k;
    const int s = (int)(c % (uint64_t)S);
    const uint32_t par = (uint32_t)((c / (uint64_t)S) & 1u);
    if (!wait_bounded_drain(&full[s], par)) atomicOr(p.err, 1u);
  }
}

// Consumers: fold each rank slice as it lands, add the residual, store ar and
// residual_out, combine the row's sum of squares (CTA, then cluster), store
// norm_out.  On a failed wait they record it and leave the row loop.
//
// With LS > 0 the last LS slices of a row (the last ranks and the residual)
// skip the ring: each consumer loads its own columns of them with 16-byte
// loads issued when the row starts, and folds them, still in rank order,
// after the bulk-copied slices.  One thread issues the bulk copies one after
// another (about 0.32 us each for 16 KB on GB300), so fewer copies per row
// shorten every row whose SM is not waiting on HBM anyway: the first row
// and the last, partial wave.
template <int DT, int W, int VPT, int LS>
__device__ __forceinline__ void run_consumers(const TmaParams& p, uint8_t* ring, uint64_t* full, uint64_t* empty,
                                              uint64_t* rowbar, uint64_t* xbar, float* s_warp, float* s_part,
                                              float* s_total, volatile int* s_abort, int S, int slice, int cols,
                                              int n, uint32_t crank, int64_t group, int64_t ngroups,
                                              int nconsumer_warps) {
  constexpr int E = Pack<DT>::kN;
  const int C = p.cluster;
  const int T = p.consumers;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col0 = (int)crank * cols;
  uint4 wv[VPT];
  bool ok_col[VPT];
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int v = threadIdx.x + k * T;
    ok_col[k] = v < cols;
    wv[k] = ok_col[k] ? __ldg(p.weight + col0 + v) : make_uint4(0u, 0u, 0u, 0u);
  }
  int slot = 0;
  uint32_t phase = 0, it = 0;
  bool failed = false;
  const int nt = n + 1 - LS;  // slices that come through the ring
  for (int64_t row = group; row < p.rows && !failed; row += ngroups, it++) {
    const int64_t rbase = row * (int64_t)p.vec_per_row + col0;
    float acc[VPT][E];
    float ss = 0.f;
    uint4 lreg[LS > 0 ? LS : 1][VPT];
    if constexpr (LS > 0) {
#pragma unroll
      for (int j = 0; j < LS; j++) {
        const int q = nt + j;
        const uint4* src = q < n ? static_cast<const uint4*>(p.in.p[q]) : reinterpret_cast<const uint4*>(p.residual);
#pragma unroll
        for (int k = 0; k < VPT; k++)
          if (ok_col[k]) lreg[j][k] = ld_stream(src + rbase + threadIdx.x + k * T);
      }
    }
    for (int q = 0; q < nt; q++) {
      if (!wait_bounded(&full[slot], phase, s_abort)) {
        failed = true;
        break;
      }
      const uint8_t* sl = ring + (size_t)slot * slice;
      if (q < n) {
        // fold rank q into the accumulators (rank order, fp32)
#pragma unroll
        for (int k = 0; k < VPT; k++) {
          if (ok_col[k]) {
            float t[E];
            Pack<DT>::widen(lds16(sl + 16 * (threadIdx.x + k * T)), t);
#pragma unroll
            for (int e = 0; e < E; e++) acc[k][e] = q == 0 ? t[e] : __fadd_rn(acc[k][e], t[e]);
          }
        }
      } else {
        // residual: h = acc + residual, first two outputs, sum of squares
#pragma unroll
        for (int k = 0; k < VPT; k++) {
          if (ok_col[k]) {
            const int v = threadIdx.x + k * T;
            float rf[E];
            Pack<DT>::widen(lds16(sl + 16 * v), rf);
            if (p.ar_out) st16(p.ar_out + rbase + v, Pack<DT>::narrow(acc[k]));
#pragma unroll
            for (int e = 0; e < E; e++) {
              acc[k][e] = __fadd_rn(acc[k][e], rf[e]);  // acc now holds h
              ss = fmaf(acc[k][e], acc[k][e], ss);
            }
            st16(p.residual_out + rbase + v, Pack<DT>::narrow(acc[k]));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (failed) break;
    if constexpr (LS > 0) {
#pragma unroll
      for (int j = 0; j < LS; j++) {
        const int q = nt + j;
#pragma unroll
        for (int k = 0; k < VPT; k++) {
          if (ok_col[k]) {
            const int v = threadIdx.x + k * T;
            float t[E];
            Pack<DT>::widen(lreg[j][k], t);
            if (q < n) {
#pragma unroll
              for (int e = 0; e < E; e++) acc[k][e] = q == 0 ? t[e] : __fadd_rn(acc[k][e], t[e]);
            } else {
              if (p.ar_out) st16(p.ar_out + rbase + v, Pack<DT>::narrow(acc[k]));
#pragma unroll
              for (int e = 0; e < E; e++) {
                acc[k][e] = __fadd_rn(acc[k][e], t[e]);  // acc now holds h
                ss = fmaf(acc[k][e], acc[k][e], ss);
              }
              st16(p.residual_out + rbase + v, Pack<DT>::narrow(acc[k]));
            }
          }
        }
      }
    }
    // row statistic: warp partials -> CTA partial -> (cluster) row total
    ss = warp_sum(ss);
    float* sw = s_warp + 16 * (it & 1u);
    if (lane == 0) {
      sw[warp] = ss;
      mbar_arrive(&rowbar[0]);
    }
    if (!wait_bounded(&rowbar[0], it & 1u, s_abort)) {
      failed = true;
      break;
    }
    // One CTA per row: every warp adds the warp partials itself (same values,
    // same order, so the same total) and the row needs no second barrier;
    // the partials are double-buffered by row parity, since a warp rewrites
    // its slot for row it + 2 only after every warp has arrived for row
    // it + 1.  Measured on GB300 at W = 8, M = 512, N = 8192 bf16 against
    // warp 0 adding them and broadcasting through rowbar[1]: 14.87 -> 14.73
    // us back to back, 25.85 -> 25.69 us per step, cold 17.49 -> 17.36 us.
    float rowtot = 0.f;
    if (C == 1) {
      rowtot = warp_sum(lane < nconsumer_warps ? sw[lane] : 0.f);
    } else {
      if (warp == 0) {
        float t = lane < nconsumer_warps ? sw[lane] : 0.f;
        t = warp_sum(t);
        int ok = 1;
        if (lane == 0) {
          // send this CTA's partial to every CTA of the cluster (itself
          // included), then add the C partials in rank order: every CTA of
          // the row gets the same total
          const uint32_t b = it & 1u;
          mbar_arrive_expect_tx(&xbar[b], 4u * (uint32_t)C);  // C partials of 4 bytes will land here
          for (int r = 0; r < C; r++)
            st_async_f32(map_rank(&s_part[2 * b + crank], (uint32_t)r), t, map_rank(&xbar[b], (uint32_t)r));
          ok = wait_bounded_cluster(&xbar[b], (it >> 1) & 1u, s_abort) ? 1 : 0;
          float tot = s_part[2 * b];
          for (int r = 1; r < C; r++) tot += s_part[2 * b + r];
          *s_total = tot;
          mbar_arrive(&rowbar[1]);
        }
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
          failed = true;
          break;
        }
      }
      if (!wait_bounded(&rowbar[1], it & 1u, s_abort)) {
        failed = true;
        break;
      }
      rowtot = *s_total;
    }
    const float rms = rsqrtf(__fdiv_rn(rowtot, p.cols) + p.eps);
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      if (ok_col[k]) {
        const int v = threadIdx.x + k * T;
        float wf[E], o[E];
        Pack<DT>::widen(wv[k], wf);
#pragma unroll
        for (int e = 0; e < E; e++) o[e] = __fmul_rn(__fmul_rn(acc[k][e], rms), wf[e]);
        st16(p.norm_out + rbase + v, Pack<DT>::narrow(o));
      }
    }
  }
  if (failed) {
    atomicOr(p.err, 1u);
    *s_abort = 1;
  }
}

template <int DT, int W, int VPT, int LS>
__global__ void __launch_bounds__(544, 1) reduce_residual_rmsnorm_tma_kernel(const TmaParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int S = p.slots;
  const int C = p.cluster;
  const int slice = p.row_bytes / C;        // bytes of one (row, rank) piece held by this CTA
  const int cols = p.vec_per_row / C;       // 16-byte columns of this CTA
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * slice);
  uint64_t* empty = full + S;
  uint64_t* rowbar = empty + S;   // [0] warp partials written, [1] row total written
  uint64_t* xbar = rowbar + 2;    // cluster rows: the CTAs' partials arrived, by row parity
  float* s_warp = reinterpret_cast<float*>(xbar + 2);   // [2][16]: 16 consumer warps at most, by row parity
  float* s_part = s_warp + 32;                           // [2][2] partials of the cluster's CTAs
  float* s_total = s_part + 4;
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_total + 1);
  volatile int* s_dep = s_abort + 1;   // set once the dependency wait has returned

  const int n = W > 0 ? W : p.nranks;
  const int nconsumer_warps = p.consumers >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = C > 1 ? cluster_rank() : 0u;
  const int64_t group = blockIdx.x / C, ngroups = gridDim.x / C;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], (uint32_t)nconsumer_warps);
    }
    mbar_init(&rowbar[0], (uint32_t)nconsumer_warps);
    mbar_init(&rowbar[1], 1);
    mbar_init(&xbar[0], 1);  // completed by the local expect_tx arrive plus C x 4 bytes
    mbar_init(&xbar[1], 1);
    *s_abort = 0;
    *s_dep = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (C > 1) cluster_barrier();  // peers' barriers exist before anyone arrives on them
  // While the previous grid of the stream finishes: this CTA's piece of its
  // first row (W ranks, residual, weight) into L2, one bulk prefetch each, by
  // the producer warp.  The first kEarlyPrefetch slices are requested at
  // once; the rest only if the dependency wait has not returned within
  // kPrefetchGraceNs, i.e. only when a previous grid is still running and
  // the prefetch can use the HBM time its tail leaves idle.  With no grid
  // before this one, prefetching the whole row only duplicates the first
  // copies and delays them.  Measured on GB300 at W = 8, M = 512, N = 8192
  // bf16 (cold launch: median of 24 ncu launches with caches flushed; step:
  // plain reduce then this kernel, graph replay).  On one box: whole row
  // always 18.03 us cold and 25.97 us per step, whole row after a 100 ns
  // grace 17.41 and 26.00.  On another: whole row after the grace 17.34 and
  // 25.68, two slices at once and the rest after the grace 17.18 and 25.54.
  // No prefetch at all: 17.07 us in graph replay of this kernel alone,
  // against 14.65 with it.  griddepcontrol.wait
  // holds the whole warp that executes it, so thread 0 (consumer warp 0)
  // waits and sets s_dep, and no lane of the producer warp waits before the
  // warp has decided.
  if (warp == nconsumer_warps && group < p.rows) {
    const int q = lane < n ? lane : 0;
    const int64_t off = group * (int64_t)p.row_bytes + (int64_t)crank * slice;
    const void* src = lane < n    ? static_cast<const void*>(static_cast<const uint8_t*>(p.in.p[q]) + off)
                      : lane == n ? static_cast<const void*>(p.residual + off)
                                  : static_cast<const void*>(p.weight + (int64_t)crank * cols);
    if (lane < kEarlyPrefetch && lane < n + 2) prefetch_l2(src, (uint32_t)slice);
    const unsigned long long t0 = globaltimer();
    while (!*s_dep && globaltimer() - t0 < kPrefetchGraceNs) {
    }
    const bool still_waiting = __any_sync(0xFFFFFFFFu, !*s_dep);
    if (still_waiting && lane >= kEarlyPrefetch && lane < n + 2) prefetch_l2(src, (uint32_t)slice);
  }
  __syncwarp();
  pdl_wait_and_release();        // inputs may come from the previous kernel of the stream
  if (threadIdx.x == 0) *s_dep = 1;

  if (warp == nconsumer_warps) {
    if (lane == 0) run_producer(p, ring, full, empty, s_abort, S, slice, n, crank, group, ngroups);
  } else {
    run_consumers<DT, W, VPT, LS>(p, ring, full, empty, rowbar, xbar, s_warp, s_part, s_total, s_abort, S, slice,
                                  cols, n, crank, group, ngroups, nconsumer_warps);
  }
  // A CTA leaves only when its cluster peer is done with its shared memory
  // (every wait above is bounded, so every thread gets here).
  if (C > 1) cluster_barrier();
}

using TmaFn = void (*)(const TmaParams);

template <int DT>
TmaFn pick_dt(int W, int vpt, int ls) {
  // register-loaded slices are used at W = 8 only (see fused_tma_shape)
  if (ls == kRegSlices) {
    if (W != 8) return nullptr;
    return vpt == 1   ? reduce_residual_rmsnorm_tma_kernel<DT, 8, 1, kRegSlices>
           : vpt == 2 ? reduce_residual_rmsnorm_tma_kernel<DT, 8, 2, kRegSlices>
                      : nullptr;
  }
  if (ls != 0) return nullptr;
#define CAR_TMA_W(WV)                                                                          \
  switch (vpt) {                                                                               \
    case 1: return reduce_residual_rmsnorm_tma_kernel<DT, WV, 1, 0>;                           \
    case 2: return reduce_residual_rmsnorm_tma_kernel<DT, WV, 2, 0>;                           \
    case 4: return reduce_residual_rmsnorm_tma_kernel<DT, WV, 4, 0>;                           \
    case 8: return reduce_residual_rmsnorm_tma_kernel<DT, WV, 8, 0>;                           \
    default: return nullptr;                                                                   \
  }
  switch (W) {
    case 2: CAR_TMA_W(2)
    case 4: CAR_TMA_W(4)
    case 8: CAR_TMA_W(8)
    case 16: CAR_TMA_W(16)
    default: CAR_TMA_W(0)
  }
#undef CAR_TMA_W
}

TmaFn pick_tma(int dtype, int W, int vpt, int ls) {
  switch (dtype) {
    case kBF16: return pick_dt<kBF16>(W, vpt, ls);
    case kFP16: return pick_dt<kFP16>(W, vpt, ls);
    default: return pick_dt<kFP32>(W, vpt, ls);
  }
}

}  // namespace

// Largest dynamic shared memory the ring may use per CTA.
constexpr int kTmaSmemBudget = 200 * 1024;

cudaError_t fused_tma_prepare(int dtype, int W, const FusedTmaShape& sh) {
  TmaFn fn = pick_tma(dtype, W, sh.vpt, sh.ls);
  if (!fn) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              sh.smem);
}

bool fused_tma_shape(int64_t rows, int vec_per_row, int num_sms, int cluster, int W, FusedTmaShape* out) {
  if (cluster != 1 && cluster != 2) return false;
  if (vec_per_row % cluster != 0) return false;
  const int cols = vec_per_row / cluster;
  const int slice = cols * 16;
  if (slice > kTmaSmemBudget / 2) return false;
  int consumers = ((cols + 31) / 32) * 32;
  if (consumers > 512) consumers = 512;
  int vpt = (cols + consumers - 1) / consumers;
  if (vpt == 3) vpt = 4;
  if (vpt > 4 && vpt <= 8) vpt = 8;
  if (vpt > 8) return false;
  // The last kRegSlices slices of a row are loaded by the consumers at W = 8
  // when a thread holds at most two vectors (register room).  Measured on
  // GB300 (N = 8192 bf16 unless noted), it pays only there: W = 8 M = 512
  // 17.4 -> 17.0 us and M = 2048 57.5 -> 55.6 us, but W = 4 (M = 512 and
  // 2048, also N = 4096 fp32), W = 6 and W = 16 were 2-10 % slower.
  const int ls = (vpt <= 2 && W == 8) ? kRegSlices : 0;
  // Ring depth: about one row's bulk-copied slices (at least 6).  Deeper
  // rings keep more bulk copies outstanding and measured slower on GB300
  // (W=8, N=8192 bf16, M=512: 17.5 us with 9 slots, 17.9 us with 12 or 18).
  int slots = W + 1 - ls < 6 ? 6 : W + 1 - ls;
  if (slots > kTmaSmemBudget / slice) slots = kTmaSmemBudget / slice;
  if (slots < 2) return false;
  const int64_t groups = num_sms / cluster;
  out->cluster = cluster;
  out->ls = ls;
  out->consumers = consumers;
  out->vpt = vpt;
  out->slots = slots;
  out->grid = (int)((rows < groups ? rows : groups) * cluster);
  out->smem = slots * slice + (2 * slots + 4) * 8 + 192;
  return true;
}

cudaError_t launch_fused_tma(int dtype, int W, const RankPtrs& in, const void* residual, const void* weight,
                             float eps, void* residual_out, void* norm_out, void* ar_out, unsigned int* err,
                             int64_t rows, int64_t cols, int vec_per_row, const FusedTmaShape& sh,
                             cudaStream_t s) {
  TmaFn fn = pick_tma(dtype, W, sh.vpt, sh.ls);
  if (!fn) return cudaErrorInvalidValue;
  TmaParams p;
  p.in = in;
  p.residual = static_cast<const uint8_t*>(residual);
  p.weight = static_cast<const uint4*>(weight);
  p.residual_out = static_cast<uint4*>(residual_out);
  p.norm_out = static_cast<uint4*>(norm_out);
  p.ar_out = static_cast<uint4*>(ar_out);
  p.err = err;
  p.eps = eps;
  p.cols = (float)cols;
  p.rows = rows;
  p.row_bytes = vec_per_row * 16;
  p.vec_per_row = vec_per_row;
  p.slots = sh.slots;
  p.tma_slices = W + 1 - sh.ls;
  p.consumers = sh.consumers;
  p.nranks = W;
  p.cluster = sh.cluster;
  return launch_pdl(fn, (unsigned)sh.grid, (unsigned)(sh.consumers + 32), (size_t)sh.smem, s,
                    (unsigned)sh.cluster, p);
}

}  // namespace car
