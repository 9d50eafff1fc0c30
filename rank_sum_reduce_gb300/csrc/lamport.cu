// lamport.cu -- Lamport one-shot push format (bf16) with the receive step
// fused with residual add + RMSNorm.
//
// P4 "用 Triton + Symmetric Memory 写一个 AllReduce + RMSNorm 融合算子",
// section "方案二：Lamport（负零轮询）": two bf16 share a 32-bit word; the
// receive buffer starts filled with the sentinel 0x80008000 (two bf16 -0.0);
// senders turn -0.0 into +0.0 so real data never equals the sentinel; the
// receiver polls its buffer until no word is the sentinel, then sums the
// ranks; buffers rotate over three regions (region = round % 3, another is
// cleared for reuse).
//
// On one GPU the receive buffer holds all W slots.  Layout: region k, slot r
// starts at byte (k * W + r) * D.  The receive kernel reads region
// round % 3, checks every word of the row against the sentinel on the same
// load, re-reads missing words at most max_polls - 1 more times (volatile),
// and refills region (round + 2) % 3 -- the previous round's -- with the
// sentinel.  Rows with a missing word in any rank are stale: their outputs
// are 0 and each (rank, row) is logged.  Roofline: HBM; a row reads
// W + 1 row slices and the weight, writes 2-3 output rows and W sentinel
// rows.
#include "car_device.cuh"
#include "car_launch.h"

namespace car {
namespace {

constexpr uint32_t kSentinel = 0x80008000u;

__global__ void __launch_bounds__(kWireThreads) lamport_fill_kernel(uint4* __restrict__ words, const int64_t nvec) {
  pdl_wait_and_release();
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += step)
    st16(words + i, make_uint4(kSentinel, kSentinel, kSentinel, kSentinel));
}

// -0.0 (0x8000) -> +0.0 in each 16-bit half; the pair layout is the data's own
__device__ __forceinline__ uint32_t scrub(uint32_t w) { return w & ~__vcmpeq2(w, kSentinel); }

__global__ void __launch_bounds__(kWireThreads)
    lamport_push_kernel(const uint4* __restrict__ data, const int64_t nvec, uint4* __restrict__ slot) {
  pdl_wait_and_release();
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += step) {
    const uint4 d = ld_stream(data + i);
    st16(slot + i, make_uint4(scrub(d.x), scrub(d.y), scrub(d.z), scrub(d.w)));
  }
}

__device__ __forceinline__ bool has_sentinel(uint4 v) {
  return v.x == kSentinel || v.y == kSentinel || v.z == kSentinel || v.w == kSentinel;
}

struct LamportParams {
  const uint8_t* region;     // slot r of the region read this round: region + r * slot_bytes
  uint8_t* clear_region;     // region refilled with the sentinel
  int64_t slot_bytes;        // D
  const uint4* residual;
  const uint4* weight;
  uint4* residual_out;
  uint4* norm_out;
  uint4* ar_out;             // may be null
  StaleLog* log;
  int log_slot;
  unsigned int* err;         // bit 0: a CTA gave up waiting for its cluster peers' partials
  float eps;
  float cols;
  int64_t rows;
  int vec_per_row;
  int chunk;
  int cluster;
  int nranks;
  int max_polls;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

template <int W, int VPT>
constexpr int max_threads() {
  return (W > 0 && W <= 4 && VPT == 1) ? 1024 : 512;
}

template <int W, int VPT>
__global__ void __launch_bounds__(max_threads<W, VPT>())
    lamport_reduce_residual_rmsnorm_kernel(const LamportParams p) {
  constexpr int E = 8;
  constexpr int R = W > 0 ? W : kMaxRanks;
  const int n = W > 0 ? W : p.nranks;
  __shared__ float s_warp[2][32];        // warp partials, by row parity
  __shared__ uint32_t s_miss_warp[2][32];  // warp masks, by row parity
  __shared__ __align__(8) uint2 s_part[2][8];  // the cluster's CTA (partial, mask) pairs, by row parity
  __shared__ __align__(8) uint64_t s_xbar[2];  // all C pairs of the row have landed, by row parity
  __shared__ float s_total;
  __shared__ uint32_t s_miss;

  const int C = p.cluster;
  const int crank = C > 1 ? (int)cluster_rank() : 0;
  const int64_t ngroups = gridDim.x / C;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int col0 = crank * p.chunk;
  uint32_t it = 0;  // rows done by this CTA
  bool peers_ready = C == 1;
  if (C > 1) {
    if (threadIdx.x == 0) {
      mbar_init(&s_xbar[0], 1);  // each phase: the local expect_tx arrive plus C x 8 bytes
      mbar_init(&s_xbar[1], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    cluster_arrive();  // its wait, before the first pair is sent, covers the loads
  }
  pdl_wait_and_release();
  prepare_next_log(p.log, p.log_slot);

  for (int64_t row = blockIdx.x / C; row < p.rows; row += ngroups, it++) {
    const int64_t rbase = row * (int64_t)p.vec_per_row;
    uint4 raw[VPT][R];
    uint4 res[VPT], wv[VPT];
    bool ok[VPT];
    uint32_t miss = 0;  // bit r: a word of rank r in this thread's columns is still the sentinel
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      const int v = threadIdx.x + k * blockDim.x;
      ok[k] = v < p.chunk && col0 + v < p.vec_per_row;
      if (ok[k]) {
        const int64_t off = (rbase + col0 + v) * 16;
#pragma unroll
        for (int r = 0; r < R; r++)
          if (r < n) raw[k][r] = ld_wire(p.region + r * p.slot_bytes + off);
        res[k] = ld_stream(p.residual + rbase + col0 + v);
        wv[k] = __ldg(p.weight + col0 + v);
      }
    }
#pragma unroll
    for (int k = 0; k < VPT; k++)
      if (ok[k])
#pragma unroll
        for (int r = 0; r < R; r++)
          if (r < n && has_sentinel(raw[k][r])) miss |= 1u << r;
    // bounded re-polls of the words still missing (volatile: each poll reaches memory)
    for (int poll = 1; poll < p.max_polls && miss; poll++) {
      uint32_t again = 0;
#pragma unroll
      for (int k = 0; k < VPT; k++) {
        if (ok[k]) {
          const int64_t off = (rbase + col0 + threadIdx.x + k * blockDim.x) * 16;
#pragma unroll
          for (int r = 0; r < R; r++) {
            if (r < n && (miss >> r & 1u)) {
              raw[k][r] = ld_wire_poll(p.region + r * p.slot_bytes + off);
              if (has_sentinel(raw[k][r])) again |= 1u << r;
            }
          }
        }
      }
      miss = again;
    }

    // rank sum in rank order, residual add, sum of squares
    float acc[VPT][E], h[VPT][E];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      if (ok[k]) {
        rank_sum<kBF16, R>(raw[k], n, acc[k]);
        float rf[E];
        Pack<kBF16>::widen(res[k], rf);
#pragma unroll
        for (int e = 0; e < E; e++) {
          h[k][e] = __fadd_rn(acc[k][e], rf[e]);
          ss = fmaf(h[k][e], h[k][e], ss);
        }
      }
    }

    // row statistic and row "missing" mask: warp -> CTA -> cluster.  One
    // CTA per row: warp 0 combines the warp pairs and broadcasts them through
    // shared memory.  Split rows: every warp combines the warp pairs itself
    // (same values, same order), lanes 0 .. C-1 of warp 0 push the CTA's
    // (partial, mask) pair into every CTA of the cluster with st.async, and
    // every thread combines the C pairs in rank order once they have landed,
    // so every CTA of the row sees the same total and mask without a second
    // CTA barrier (as in the fused row kernel).
    ss = warp_sum(ss);
    miss = __reduce_or_sync(0xFFFFFFFFu, miss);
    const uint32_t b = it & 1u;
    if (lane == 0) {
      s_warp[b][warp] = ss;
      s_miss_warp[b][warp] = miss;
    }
    if (!peers_ready) {
      cluster_wait();  // every peer's mbarriers are initialised
      peers_ready = true;
    }
    __syncthreads();
    float total;
    uint32_t row_miss;
    if (C == 1) {
      if (warp == 0) {
        const float t = warp_sum(lane < nwarps ? s_warp[b][lane] : 0.f);
        const uint32_t m = __reduce_or_sync(0xFFFFFFFFu, lane < nwarps ? s_miss_warp[b][lane] : 0u);
        if (lane == 0) {
          s_total = t;
          s_miss = m;
        }
      }
      __syncthreads();
      total = s_total;
      row_miss = s_miss;
    } else {
      // s_warp[b], s_miss_warp[b], s_part[b] and s_xbar[b] are next written
      // for row it + 2, after this CTA's first barrier of row it + 1.
      float t = warp_sum(lane < nwarps ? s_warp[b][lane] : 0.f);
      uint32_t m = __reduce_or_sync(0xFFFFFFFFu, lane < nwarps ? s_miss_warp[b][lane] : 0u);
      if (warp == 0) {
        // every lane holds the same (t, m); lane r pushes it to CTA r
        if (lane == 0) mbar_arrive_expect_tx(&s_xbar[b], 8u * (uint32_t)C);
        if (lane < C)
          st_async_v2_b32(map_rank(&s_part[b][crank], (uint32_t)lane), __float_as_uint(t), m,
                          map_rank(&s_xbar[b], (uint32_t)lane));
      }
      if (wait_cluster_phase(&s_xbar[b], (it >> 1) & 1u)) {
        t = __uint_as_float(s_part[b][0].x);
        m = s_part[b][0].y;
        for (int r = 1; r < C; r++) {
          t += __uint_as_float(s_part[b][r].x);
          m |= s_part[b][r].y;
        }
      } else {
        atomicOr(p.err, 1u);
        m = (1u << n) - 1u;  // the row's outputs are zeroed and every rank is logged for it
        // Late partials may still land: wait for them (bounded again) so
        // that none reaches this CTA's shared memory after it has exited.
        if (!wait_cluster_phase(&s_xbar[b], (it >> 1) & 1u)) atomicOr(p.err, 2u);
      }
      total = t;
      row_miss = m;
    }
    if (row_miss && crank == 0 && threadIdx.x == 0) {
      for (int r = 0; r < n; r++)
        if (row_miss >> r & 1u) log_stale(p.log, p.log_slot, (uint32_t)r, (uint32_t)row);
    }
    const float rms = rsqrtf(__fdiv_rn(total, p.cols) + p.eps);
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      if (ok[k]) {
        const int v = col0 + threadIdx.x + k * blockDim.x;
        uint4 o_ar = make_uint4(0u, 0u, 0u, 0u), o_res = o_ar, o_norm = o_ar;
        if (!row_miss) {
          float wf[E], o[E];
          Pack<kBF16>::widen(wv[k], wf);
#pragma unroll
          for (int e = 0; e < E; e++) o[e] = __fmul_rn(__fmul_rn(h[k][e], rms), wf[e]);
          o_ar = Pack<kBF16>::narrow(acc[k]);
          o_res = Pack<kBF16>::narrow(h[k]);
          o_norm = Pack<kBF16>::narrow(o);
        }
        if (p.ar_out) st16(p.ar_out + rbase + v, o_ar);
        st16(p.residual_out + rbase + v, o_res);
        st16(p.norm_out + rbase + v, o_norm);
        // refill the previous round's region at the same place in every slot
        const int64_t off = (rbase + v) * 16;
        const uint4 sent = make_uint4(kSentinel, kSentinel, kSentinel, kSentinel);
        for (int r = 0; r < n; r++) st16(p.clear_region + r * p.slot_bytes + off, sent);
      }
    }
  }
  // Nothing reaches this CTA's shared memory after its last row's wait (each
  // peer sends one pair per row), so no exit barrier is needed; a cluster with
  // no row still pairs its first arrive.
  if (!peers_ready) cluster_wait();
}

using LamportFn = void (*)(const LamportParams);

LamportFn pick_lamport(int W, int vpt) {
  if (vpt == 2) {
    switch (W) {
      case 2: return lamport_reduce_residual_rmsnorm_kernel<2, 2>;
      case 4: return lamport_reduce_residual_rmsnorm_kernel<4, 2>;
      case 8: return lamport_reduce_residual_rmsnorm_kernel<8, 2>;
      default: return nullptr;
    }
  }
  if (vpt != 1) return nullptr;
  switch (W) {
    case 2: return lamport_reduce_residual_rmsnorm_kernel<2, 1>;
    case 4: return lamport_reduce_residual_rmsnorm_kernel<4, 1>;
    case 8: return lamport_reduce_residual_rmsnorm_kernel<8, 1>;
    case 16: return lamport_reduce_residual_rmsnorm_kernel<16, 1>;
    default: return lamport_reduce_residual_rmsnorm_kernel<0, 1>;
  }
}

}  // namespace

bool lamport_has_variant(int W, int vpt) {
  if (vpt == 1) return true;
  return vpt == 2 && (W == 2 || W == 4 || W == 8);
}

int lamport_max_threads(int W, int vpt) { return (vpt == 1 && (W == 2 || W == 4)) ? 1024 : 512; }

cudaError_t lamport_resident_groups(int W, const FusedShape& sh, int num_sms, int* groups) {
  *groups = 0;
  LamportFn fn = pick_lamport(W, sh.vpt);
  if (!fn) return cudaErrorInvalidValue;
  if (sh.cluster == 1) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void*>(fn),
                                                                  sh.threads, 0);
    if (e != cudaSuccess) return e;
    *groups = per_sm * num_sms;
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sh.cluster, 1, 1);
  cfg.blockDim = dim3((unsigned)sh.threads, 1, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)sh.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(groups, reinterpret_cast<const void*>(fn), &cfg);
}

cudaError_t launch_lamport_fill(void* words, int64_t bytes, int grid, cudaStream_t s) {
  return launch_pdl(lamport_fill_kernel, (unsigned)grid, kWireThreads, 0, s, 1, static_cast<uint4*>(words),
                    bytes / 16);
}

cudaError_t launch_lamport_push(const void* data, int64_t bytes, void* slot, int grid, cudaStream_t s) {
  return launch_pdl(lamport_push_kernel, (unsigned)grid, kWireThreads, 0, s, 1, static_cast<const uint4*>(data),
                    bytes / 16, static_cast<uint4*>(slot));
}

cudaError_t launch_lamport_reduce(int W, const void* region, void* clear_region, int64_t slot_bytes,
                                  const void* residual, const void* weight, float eps, void* residual_out,
                                  void* norm_out, void* ar_out, StaleLog* log, int log_slot, int max_polls,
                                  unsigned int* err, int64_t rows, int64_t cols, int vec_per_row,
                                  const FusedShape& sh, cudaStream_t s) {
  LamportFn fn = pick_lamport(W, sh.vpt);
  if (!fn) return cudaErrorInvalidValue;
  LamportParams p;
  p.region = static_cast<const uint8_t*>(region);
  p.clear_region = static_cast<uint8_t*>(clear_region);
  p.slot_bytes = slot_bytes;
  p.residual = static_cast<const uint4*>(residual);
  p.weight = static_cast<const uint4*>(weight);
  p.residual_out = static_cast<uint4*>(residual_out);
  p.norm_out = static_cast<uint4*>(norm_out);
  p.ar_out = static_cast<uint4*>(ar_out);
  p.log = log;
  p.log_slot = log_slot;
  p.err = err;
  p.eps = eps;
  p.cols = (float)cols;
  p.rows = rows;
  p.vec_per_row = vec_per_row;
  p.chunk = (vec_per_row + sh.cluster - 1) / sh.cluster;
  p.cluster = sh.cluster;
  p.nranks = W;
  p.max_polls = max_polls;
  return launch_pdl(fn, (unsigned)(sh.groups * sh.cluster), (unsigned)sh.threads, 0, s, (unsigned)sh.cluster, p);
}

}  // namespace car
