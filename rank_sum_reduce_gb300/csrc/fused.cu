// fused.cu -- rank sum + residual add + RMSNorm in one pass over HBM.
//
// P4 "用 Triton + Symmetric Memory 写一个 AllReduce + RMSNorm 融合算子",
// sections "这个算子在算什么" (ar = sum_r x_r; h = ar + residual;
// rms = rsqrt(mean(h^2) + eps); out = (h * rms) * weight) and "总体设计"
// (read every rank's row, fp32 sum, add residual and store residual_out, then
// mean of squares, rsqrt, scale by weight and store norm_out, while the sum is
// still in registers).  The rank sum itself follows P1
// "1stage：kernel 全文与时间线" (fixed rank order, fp32, one rounding).
//
// GB300 design, differing from the page: the page gives a whole row to one
// program and leaves the rest of the GPU idle at M = 1.  Here a row can be
// split over a thread-block cluster of up to 8 CTAs on different SMs; each CTA
// reduces its slice and pushes its partial sum of squares into every peer's
// shared memory (st.async, counted on the peer's mbarrier), so the row's total
// is one one-way hop away.  With many rows, one CTA takes a row and CTAs loop
// over rows (grid capped at the resident count).  Each CTA's first row is
// requested into L2 before the PDL wait.  h never leaves registers.
// Roofline: HBM, (W + 1 + outputs) * 16 bytes per vector plus the weight row.
#include "car_device.cuh"
#include "car_launch.h"

namespace car {
namespace {

struct FusedParams {
  RankPtrs in;
  const uint4* residual;
  const uint4* weight;
  uint4* residual_out;
  uint4* norm_out;
  uint4* ar_out;  // may be null
  unsigned int* err;  // bit 0: a CTA gave up waiting for its cluster peers' partials
  float eps;
  float cols;     // N, exactly representable (N <= 2^24)
  int64_t rows;
  int vec_per_row;
  int chunk;      // 16-byte vectors of a row handled by one CTA
  int cluster;    // CTAs per row
  int nranks;
  // The bounded wait for a split row's partials, and a test hook that holds
  // back one CTA's partial (see car_test_delay_partial): CTA `delay_cta` of
  // the cluster that takes row `delay_row` pushes its partial `delay_ns`
  // late.  delay_cta < 0: no delay.
  unsigned long long wait_ns;
  unsigned long long delay_ns;
  int64_t delay_row;
  int delay_cta;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Ask L2 for this CTA's piece of `row` -- the n rank slices, the residual and,
// when `weight`, the weight -- with one bulk prefetch per slice, issued by
// threads 0 .. n (+1).  L2 is coherent for the whole GPU, so this may run
// before the PDL wait.
__device__ __forceinline__ void prefetch_row(const FusedParams& p, int n, int64_t row, int col0, bool weight) {
  const int nvec = min(p.chunk, p.vec_per_row - col0);
  const int t = threadIdx.x;
  if (row >= p.rows || nvec <= 0 || t > n + (weight ? 1 : 0)) return;
  const int64_t off = row * (int64_t)p.vec_per_row + col0;
  const uint4* src = t < n ? static_cast<const uint4*>(p.in.p[t]) + off : (t == n ? p.residual + off : p.weight + col0);
  prefetch_l2(src, (uint32_t)nvec * 16u);
}

template <int W, int VPT>
constexpr int max_threads() {
  return (W > 0 && W <= 4 && VPT == 1) ? 1024 : 512;
}

// MINB: CTAs per SM the instance is compiled for.  W = 8 with one vector per
// thread has a second instance held to two 512-thread CTAs per SM (64
// registers, no spills) for one CTA per row over many rows, where a second
// resident row pays: N = 4096 bf16, M = 256 5.40 -> 4.70 us, M = 1024 15.5 ->
// 14.7 us.  Split rows keep the unbounded instance, whose latency is lower
// (W = 8, M = 1, N = 8192: 1.92 against 2.02 us).
template <int DT, int W, int VPT, int MINB>
__global__ void __launch_bounds__(max_threads<W, VPT>(), MINB)
    reduce_residual_rmsnorm_kernel(const FusedParams p) {
  constexpr int E = Pack<DT>::kN;
  constexpr int R = W > 0 ? W : kMaxRanks;
  const int n = W > 0 ? W : p.nranks;
  __shared__ float s_warp[2][32];             // warp partials, by row parity
  __shared__ float s_part[2][8];               // the cluster's CTA partials, by row parity
  __shared__ __align__(8) uint64_t s_xbar[2];  // all C partials of the row have landed, by row parity
  __shared__ float s_total;

  // Instances held to two CTAs per SM are launched for whole rows only.
  const int C = MINB > 1 ? 1 : p.cluster;
  const int crank = C > 1 ? (int)cluster_rank() : 0;
  const int64_t ngroups = gridDim.x / C;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int col0 = crank * p.chunk;
  uint32_t it = 0;  // rows done by this CTA
  bool peers_ready = C == 1;
  if (C > 1) {
    if (threadIdx.x == 0) {
      mbar_init(&s_xbar[0], 1);  // each phase: the local expect_tx arrive plus C x 4 bytes
      mbar_init(&s_xbar[1], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    cluster_arrive();  // its wait, before the first partial is sent, covers the loads
  }
  // While the previous grid of the stream finishes: this CTA's first row.
  prefetch_row(p, n, blockIdx.x / C, col0, true);
  pdl_wait_and_release();

  for (int64_t row = blockIdx.x / C; row < p.rows; row += ngroups, it++) {
    const int64_t rbase = row * (int64_t)p.vec_per_row;
    // With more rows than CTAs: this CTA's next row while this one is reduced.
    // Many rows of 8 KB and less: W = 4, M = 1024, N = 4096 bf16 11.8 -> 10.1
    // us; M = 4096 38.4 -> 34.8 us; W = 2, M = 4096, N = 1024 8.9 -> 7.6 us.
    prefetch_row(p, n, row + ngroups, col0, false);

    // 1. all loads of this thread's vectors: W ranks + residual
    uint4 raw[VPT][R];
    uint4 res[VPT], wv[VPT];
    bool ok[VPT];
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      const int v = threadIdx.x + k * blockDim.x;
      ok[k] = v < p.chunk && col0 + v < p.vec_per_row;
      if (ok[k]) {
        const int64_t off = rbase + col0 + v;
#pragma unroll
        for (int r = 0; r < R; r++)
          if (r < n) raw[k][r] = ld_stream(static_cast<const uint4*>(p.in.p[r]) + off);
        res[k] = ld_stream(p.residual + off);
        wv[k] = __ldg(p.weight + col0 + v);  // issued with the inputs: off the statistic's critical path
      }
    }

    // 2. rank sum, residual add, first two outputs, sum of squares
    float h[VPT][E];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      if (ok[k]) {
        const int64_t off = rbase + col0 + threadIdx.x + k * blockDim.x;
        float acc[E];
        rank_sum<DT, R>(raw[k], n, acc);
        if (p.ar_out) st16(p.ar_out + off, Pack<DT>::narrow(acc));
        float rf[E];
        Pack<DT>::widen(res[k], rf);
#pragma unroll
        for (int e = 0; e < E; e++) {
          h[k][e] = __fadd_rn(acc[e], rf[e]);
          ss = fmaf(h[k][e], h[k][e], ss);
        }
        st16(p.residual_out + off, Pack<DT>::narrow(h[k]));
      }
    }

    // 3. row statistic: warp shuffle, then shared memory across warps.
    //    One CTA per row: warp 0 adds the warp partials and broadcasts the
    //    total through shared memory.  Split rows: every warp adds the warp
    //    partials itself (same values, same order, so the same sum), lanes
    //    0 .. C-1 of warp 0 push it into every CTA of the cluster (st.async,
    //    counted on the receiver's mbarrier), and every thread waits for the
    //    C partials and adds them in rank order: one one-way hop, no second
    //    CTA barrier, and every CTA of the row sees the same total.  The
    //    butterfly leaves the same sum in every lane (at each step both lanes
    //    of a pair add the same two values, in either order, and fp32
    //    addition commutes).  Back to back, W = 8, M = 1, N = 8192: 2.01 ->
    //    1.96 us per call from pushing with C lanes instead of one, then
    //    1.95 -> 1.84 us (another box) from dropping the second barrier;
    //    W = 16: 2.08 -> 1.98 us.  With one CTA per row the second barrier
    //    stays: every warp adding the partials itself there made many rows
    //    per CTA 1-2 % slower.
    ss = warp_sum(ss);
    const uint32_t b = it & 1u;
    if (lane == 0) s_warp[b][warp] = ss;
    if (!peers_ready) {
      cluster_wait();  // every peer's mbarriers are initialised
      peers_ready = true;
    }
    // test hook: this whole CTA reaches the exchange late
    if (C > 1 && crank == p.delay_cta && row == p.delay_row) spin_ns(p.delay_ns);
    __syncthreads();
    float total;
    if (C == 1) {
      if (warp == 0) {
        const float t = warp_sum(lane < nwarps ? s_warp[b][lane] : 0.f);
        if (lane == 0) s_total = t;
      }
      __syncthreads();
      total = s_total;
    } else {
      // s_warp[b], s_part[b] and s_xbar[b] are next written for row it + 2,
      // after this CTA's first barrier of row it + 1, which every thread
      // reaches only once it has read them for this row.
      float t = warp_sum(lane < nwarps ? s_warp[b][lane] : 0.f);
      const uint32_t par = (it >> 1) & 1u;
      if (warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(&s_xbar[b], 4u * (uint32_t)C);
        if (lane < C)
          st_async_f32(map_rank(&s_part[b][crank], (uint32_t)lane), t, map_rank(&s_xbar[b], (uint32_t)lane));
      }
      if (wait_cluster_phase(&s_xbar[b], par, p.wait_ns)) {
        t = s_part[b][0];
        for (int r = 1; r < C; r++) t += s_part[b][r];
      } else {
        atomicOr(p.err, 1u);
        t = __int_as_float(0x7fc00000);  // NaN: this row's norm_out is not usable
        // The missing partials may still come: wait (bounded again) until
        // they have landed, so that none reaches this CTA's shared memory
        // after it has exited and the barrier's phases stay in step for the
        // next row.
        if (!wait_cluster_phase(&s_xbar[b], par)) atomicOr(p.err, 2u);
      }
      total = t;
    }
    const float rms = rsqrtf(__fdiv_rn(total, p.cols) + p.eps);

    // 4. normalise and scale
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      if (ok[k]) {
        const int col = col0 + threadIdx.x + k * blockDim.x;
        float wf[E];
        Pack<DT>::widen(wv[k], wf);
        float o[E];
#pragma unroll
        for (int e = 0; e < E; e++) o[e] = __fmul_rn(__fmul_rn(h[k][e], rms), wf[e]);
        st16(p.norm_out + rbase + col, Pack<DT>::narrow(o));
      }
    }
  }
  // Nothing reaches this CTA's shared memory after its last row's wait (each
  // peer sends one partial per row), so no exit barrier is needed; a cluster
  // with no row still pairs its first arrive.
  if (!peers_ready) cluster_wait();
}

using FusedFn = void (*)(const FusedParams);

template <int DT>
FusedFn pick_dt(int W, int vpt, int cluster) {
  if (vpt == 2) {
    switch (W) {
      case 1: return reduce_residual_rmsnorm_kernel<DT, 1, 2, 1>;
      case 2: return reduce_residual_rmsnorm_kernel<DT, 2, 2, 1>;
      case 4: return reduce_residual_rmsnorm_kernel<DT, 4, 2, 1>;
      case 8: return reduce_residual_rmsnorm_kernel<DT, 8, 2, 1>;
      default: return nullptr;
    }
  }
  if (vpt != 1) return nullptr;
  switch (W) {
    case 1: return reduce_residual_rmsnorm_kernel<DT, 1, 1, 1>;
    case 2: return reduce_residual_rmsnorm_kernel<DT, 2, 1, 1>;
    case 4: return reduce_residual_rmsnorm_kernel<DT, 4, 1, 1>;
    case 8: return cluster == 1 ? reduce_residual_rmsnorm_kernel<DT, 8, 1, 2> : reduce_residual_rmsnorm_kernel<DT, 8, 1, 1>;
    case 16: return reduce_residual_rmsnorm_kernel<DT, 16, 1, 1>;
    default: return reduce_residual_rmsnorm_kernel<DT, 0, 1, 1>;
  }
}

FusedFn pick_fused(int dtype, int W, int vpt, int cluster) {
  switch (dtype) {
    case kBF16: return pick_dt<kBF16>(W, vpt, cluster);
    case kFP16: return pick_dt<kFP16>(W, vpt, cluster);
    default: return pick_dt<kFP32>(W, vpt, cluster);
  }
}

cudaLaunchConfig_t make_config(const FusedShape& sh, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sh.groups * sh.cluster), 1, 1);
  cfg.blockDim = dim3((unsigned)sh.threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)sh.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = sh.cluster > 1 ? 1 : 0;
  return cfg;
}

}  // namespace

int fused_max_threads(int W, int vpt) {
  // W outside {1, 2, 4, 8, 16} runs the runtime-W instance, compiled for 512.
  const bool compiled_w = W == 1 || W == 2 || W == 4;
  return (vpt == 1 && compiled_w) ? 1024 : 512;
}

bool fused_has_variant(int W, int vpt) {
  if (vpt == 1) return true;
  return vpt == 2 && (W == 1 || W == 2 || W == 4 || W == 8);
}

cudaError_t fused_resident_groups(int dtype, int W, const FusedShape& sh, int num_sms, int* groups) {
  *groups = 0;
  FusedFn fn = pick_fused(dtype, W, sh.vpt, sh.cluster);
  if (!fn) return cudaErrorInvalidValue;
  if (sh.cluster == 1) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, reinterpret_cast<const void*>(fn), sh.threads, 0);
    if (e != cudaSuccess) return e;
    *groups = per_sm * num_sms;
    return cudaSuccess;
  }
  cudaLaunchAttribute attr[1];
  FusedShape probe = sh;
  probe.groups = 1;
  cudaLaunchConfig_t cfg = make_config(probe, 0, attr);
  int clusters = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void*>(fn), &cfg);
  if (e != cudaSuccess) return e;
  *groups = clusters;
  return cudaSuccess;
}

cudaError_t launch_fused(int dtype, int W, const RankPtrs& in, const void* residual,
                         const void* weight, float eps, void* residual_out, void* norm_out,
                         void* ar_out, unsigned int* err, int64_t rows, int64_t cols, int vec_per_row,
                         const FusedShape& sh, const WaitHook& hook, cudaStream_t s) {
  FusedFn fn = pick_fused(dtype, W, sh.vpt, sh.cluster);
  if (!fn) return cudaErrorInvalidValue;
  FusedParams p;
  p.in = in;
  p.residual = static_cast<const uint4*>(residual);
  p.weight = static_cast<const uint4*>(weight);
  p.residual_out = static_cast<uint4*>(residual_out);
  p.norm_out = static_cast<uint4*>(norm_out);
  p.ar_out = static_cast<uint4*>(ar_out);
  p.err = err;
  p.eps = eps;
  p.cols = (float)cols;
  p.rows = rows;
  p.vec_per_row = vec_per_row;
  p.chunk = (vec_per_row + sh.cluster - 1) / sh.cluster;
  p.cluster = sh.cluster;
  p.nranks = W;
  p.wait_ns = hook.wait_ns;
  p.delay_ns = hook.delay_ns;
  p.delay_row = hook.delay_row;
  p.delay_cta = hook.delay_cta;
  return launch_pdl(fn, (unsigned)(sh.groups * sh.cluster), (unsigned)sh.threads, 0, s, (unsigned)sh.cluster, p);
}

}  // namespace car
