// reduce.cu -- one-shot rank sum of W rank buffers held in HBM.
//
// P1 "SGLang Custom AllReduce v1 线程模型和工作原理细节", section
// "1stage：kernel 全文与时间线" (packed_reduce: upcast rank 0, add ranks
// 1..W-1 in order in fp32, downcast once) and P3 "0-custom-all-reduce",
// sections "2. 线程怎么分活" / "3. 从所有 GPU 读" (grid-stride over 16-byte
// vectors, all W loads unrolled so they are in flight together).
//
// GB300 design, differing from the pages: the grid is sized to the message
// and capped at the resident CTA count of the 152 SMs (no 36-block cap), every
// thread keeps U x W independent 16-byte loads in flight, and the rank inputs
// come from local HBM instead of NVLink peers, so there is no entry or exit
// barrier.  Each CTA takes one contiguous, equal share of the vectors (within
// one), so all CTAs finish together; a grid-stride loop over fixed waves of
// grid * threads * U vectors leaves part of the grid idle in the last wave
// (8 MB per rank at W = 8 is 3.37 waves).  Roofline: HBM, (W + 1) * 16 bytes
// per vector.
#include "car_device.cuh"
#include "car_launch.h"

namespace car {
namespace {

// This CTA's share [lo, hi) of the vectors: nvec / grid, one more for the
// first nvec % grid CTAs.
__device__ __forceinline__ void cta_share(const int64_t nvec, int64_t* lo, int64_t* hi) {
  const int64_t share = nvec / gridDim.x, extra = nvec % gridDim.x;
  *lo = share * blockIdx.x + (blockIdx.x < extra ? blockIdx.x : extra);
  *hi = *lo + share + (blockIdx.x < extra ? 1 : 0);
}

// Called before the PDL wait, while the previous grid of the stream
// finishes: the first pass (kReduceThreads * U vectors) of the share, every
// rank, into L2, one request per 128-byte line (a line's first vector, and
// the pass's first vector).  Per-thread requests, not bulk ones: a bulk
// prefetch per rank measured slower, alone and after the fused kernel.
template <int R, int U>
__device__ __forceinline__ void prefetch_first_pass(const RankPtrs& in, const int n, const int64_t lo,
                                                    const int64_t hi) {
#pragma unroll
  for (int u = 0; u < U; u++) {
    const int64_t v = lo + threadIdx.x + (int64_t)u * kReduceThreads;
    if (v < hi) {
#pragma unroll
      for (int r = 0; r < R; r++) {
        const uint4* a = static_cast<const uint4*>(in.p[r]) + v;
        if (r < n && ((threadIdx.x == 0 && u == 0) || (reinterpret_cast<uintptr_t>(a) & 127) == 0)) prefetch_line_l2(a);
      }
    }
  }
}

template <int DT, int W, int U>
__global__ void __launch_bounds__(kReduceThreads)
    rank_sum_reduce_kernel(const RankPtrs in, const int nranks, uint4* __restrict__ out,
                           const int64_t nvec) {
  constexpr int R = W > 0 ? W : kMaxRanks;
  const int n = W > 0 ? W : nranks;
  int64_t lo, hi;
  cta_share(nvec, &lo, &hi);
  prefetch_first_pass<R, U>(in, n, lo, hi);
  pdl_wait_and_release();
  for (int64_t base = lo + threadIdx.x; base < hi; base += kReduceThreads * U) {
    uint4 raw[U][R];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int64_t v = base + (int64_t)u * kReduceThreads;
      if (v < hi) {
#pragma unroll
        for (int r = 0; r < R; r++)
          if (r < n) raw[u][r] = ld_stream(static_cast<const uint4*>(in.p[r]) + v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int64_t v = base + (int64_t)u * kReduceThreads;
      if (v < hi) {
        float acc[Pack<DT>::kN];
        rank_sum<DT, R>(raw[u], n, acc);
        st16(out + v, Pack<DT>::narrow(acc));
      }
    }
  }
}

// Two-shot bit pattern (P1 "2stage：分片、轮转、以及为什么没有出口 barrier"):
// the 16-byte units are cut into W shards of `part` units (the last shard
// takes the remainder, and everything when part == 0); shard s is summed in
// the rotated order s, s+1, ..., s-1.  On one GPU there is nothing to
// scatter or gather: the kernel reproduces the owner's rounding in one pass.
template <int DT, int W, int U>
__global__ void __launch_bounds__(kReduceThreads)
    rank_sum_two_shot_kernel(const RankPtrs in, const int nranks, uint4* __restrict__ out,
                             const int64_t nvec, const int64_t part) {
  constexpr int R = W > 0 ? W : kMaxRanks;
  const int n = W > 0 ? W : nranks;
  // the pointer table, indexed by a per-vector rank: shared memory instead of a local copy
  __shared__ const uint4* s_ptr[kMaxRanks];
  if (threadIdx.x == 0) {
#pragma unroll
    for (int r = 0; r < kMaxRanks; r++) s_ptr[r] = static_cast<const uint4*>(in.p[r]);
  }
  __syncthreads();
  int64_t lo, hi;
  cta_share(nvec, &lo, &hi);
  prefetch_first_pass<R, U>(in, n, lo, hi);
  pdl_wait_and_release();
  for (int64_t base = lo + threadIdx.x; base < hi; base += kReduceThreads * U) {
    uint4 raw[U][R];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int64_t v = base + (int64_t)u * kReduceThreads;
      if (v < hi) {
        int owner = n - 1;
        if (part > 0 && v / part < n - 1) owner = (int)(v / part);
#pragma unroll
        for (int i = 0; i < R; i++) {
          if (i < n) {
            int r = owner + i;
            if (r >= n) r -= n;
            raw[u][i] = ld_stream(s_ptr[r] + v);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int64_t v = base + (int64_t)u * kReduceThreads;
      if (v < hi) {
        float acc[Pack<DT>::kN];
        rank_sum<DT, R>(raw[u], n, acc);
        st16(out + v, Pack<DT>::narrow(acc));
      }
    }
  }
}

using ReduceFn = void (*)(const RankPtrs, const int, uint4*, const int64_t);
using TwoShotFn = void (*)(const RankPtrs, const int, uint4*, const int64_t, const int64_t);

// Vectors per thread per iteration (U), so that each thread keeps 8 to 32
// 16-byte loads in flight.  Measured on GB300 with equal shares and the
// first-pass prefetch (graph replay over cold inputs, bf16, N = 8192): W = 2
// is fastest with 4 (4.13 us at 8 MiB per rank; 5.58 with 1), W = 4 with 4
// (14.0 against 14.3 us with 2 at 16 MiB), W = 16 with 2 (11.3 against
// 13.2 us with 1 at 4 MiB; 4 and 8 were slower).  W = 8 keeps 1: with 2 it
// ran 2 % faster alone in one buffer layout but made the reduce + fused step
// slower in another (26.33 against 25.94 us).
constexpr int vectors_for(int W) { return W <= 4 ? 4 : (W == 16 ? 2 : 1); }

template <int DT>
ReduceFn pick(int W) {
  switch (W) {
    case 1: return rank_sum_reduce_kernel<DT, 1, vectors_for(1)>;
    case 2: return rank_sum_reduce_kernel<DT, 2, vectors_for(2)>;
    case 4: return rank_sum_reduce_kernel<DT, 4, vectors_for(4)>;
    case 8: return rank_sum_reduce_kernel<DT, 8, vectors_for(8)>;
    case 16: return rank_sum_reduce_kernel<DT, 16, vectors_for(16)>;
    default: return rank_sum_reduce_kernel<DT, 0, 1>;
  }
}

template <int DT>
TwoShotFn pick2(int W) {
  switch (W) {
    case 1: return rank_sum_two_shot_kernel<DT, 1, vectors_for(1)>;
    case 2: return rank_sum_two_shot_kernel<DT, 2, vectors_for(2)>;
    case 4: return rank_sum_two_shot_kernel<DT, 4, vectors_for(4)>;
    case 8: return rank_sum_two_shot_kernel<DT, 8, vectors_for(8)>;
    case 16: return rank_sum_two_shot_kernel<DT, 16, vectors_for(16)>;
    default: return rank_sum_two_shot_kernel<DT, 0, 1>;
  }
}

TwoShotFn pick_two_shot(int dtype, int W) {
  switch (dtype) {
    case kBF16: return pick2<kBF16>(W);
    case kFP16: return pick2<kFP16>(W);
    default: return pick2<kFP32>(W);
  }
}

ReduceFn pick_reduce(int dtype, int W) {
  switch (dtype) {
    case kBF16: return pick<kBF16>(W);
    case kFP16: return pick<kFP16>(W);
    default: return pick<kFP32>(W);
  }
}

}  // namespace

int reduce_vectors_per_thread(int W) {
  return (W == 1 || W == 2 || W == 4 || W == 8 || W == 16) ? vectors_for(W) : 1;
}

cudaError_t reduce_occupancy(int dtype, int W, int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      blocks_per_sm, reinterpret_cast<const void*>(pick_reduce(dtype, W)), kReduceThreads, 0);
}

cudaError_t two_shot_occupancy(int dtype, int W, int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      blocks_per_sm, reinterpret_cast<const void*>(pick_two_shot(dtype, W)), kReduceThreads, 0);
}

cudaError_t launch_two_shot(int dtype, int W, const RankPtrs& in, void* out, int64_t nvec, int grid,
                            cudaStream_t s) {
  return launch_pdl(pick_two_shot(dtype, W), (unsigned)grid, kReduceThreads, 0, s, 1, in, W,
                    static_cast<uint4*>(out), nvec, nvec / W);
}

cudaError_t launch_reduce(int dtype, int W, const RankPtrs& in, void* out, int64_t nvec, int grid,
                          cudaStream_t s) {
  return launch_pdl(pick_reduce(dtype, W), (unsigned)grid, kReduceThreads, 0, s, 1, in, W,
                    static_cast<uint4*>(out), nvec);
}

}  // namespace car
