// car_device.cuh -- device-side building blocks shared by libcar's kernels:
// the rank pointer table, 16-byte loads, exact widening of packed bf16/fp16
// to fp32, and the round-to-nearest-even narrowing (CUDA's cvt intrinsics).
//
// Pages (title, then section):
//   P1 "SGLang Custom AllReduce v1 线程模型和工作原理细节"
//   P3 "0-custom-all-reduce" (SGLang JIT custom all-reduce notes)
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace car {

constexpr int kMaxRanks = 16;  // P3 "调用": kMaxNumGPU raised to 16

// W input pointers, passed by value in the kernel parameter block (128 B).
// P1 "一次调用给 kernel 什么：参数与 grid" passes its table by pointer only so
// that a captured graph can be back-filled; a single process has no such need.
struct RankPtrs {
  const void* p[kMaxRanks];
};

enum Dtype : int { kBF16 = 0, kFP16 = 1, kFP32 = 2 };

// ---------------------------------------------------------------------------
// 16-byte loads.  P1 "线程模型：16 字节一个单位": one thread moves 16 bytes
// per instruction, the widest single global access.
// ---------------------------------------------------------------------------

// Read-only streaming load: rank inputs and the residual are read exactly once
// per launch, so they bypass L1 allocation.  Safe with the documented aliasing
// (output == one input): an address is read before the same thread writes it,
// and never read again.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Coherent (non read-only path) 16-byte load for wire lines, which a producer
// may be writing while a bounded poll looks at them.
__device__ __forceinline__ uint4 ld_wire(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Re-read for a poll: volatile, so every poll reaches the memory system.
__device__ __forceinline__ uint4 ld_wire_poll(const void* p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

__device__ __forceinline__ uint64_t lo64(uint4 v) { return (uint64_t)v.x | ((uint64_t)v.y << 32); }
__device__ __forceinline__ uint64_t hi64(uint4 v) { return (uint64_t)v.z | ((uint64_t)v.w << 32); }
__device__ __forceinline__ uint4 make16(uint64_t lo, uint64_t hi) {
  return make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
}

// ---------------------------------------------------------------------------
// Packed element types: a 16-byte vector holds 8 bf16/fp16 or 4 fp32 values.
// Element 2k sits in the low half of 32-bit word k (little-endian layout).
// Widening is exact; narrowing rounds to nearest, ties to even, with
// subnormals kept (P1 "1stage：kernel 全文与时间线": upcast, accumulate in
// fp32, one downcast; P3 "4. 求和": __float22bfloat162_rn).
// ---------------------------------------------------------------------------
template <int DT>
struct Pack;

template <>
struct Pack<kBF16> {
  static constexpr int kN = 8;
  __device__ __forceinline__ static void widen(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static uint4 narrow(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const __nv_bfloat162 b = __float22bfloat162_rn(make_float2(f[2 * i], f[2 * i + 1]));
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Pack<kFP16> {
  static constexpr int kN = 8;
  __device__ __forceinline__ static void widen(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static uint4 narrow(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const __half2 b = __float22half2_rn(make_float2(f[2 * i], f[2 * i + 1]));
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Pack<kFP32> {
  static constexpr int kN = 4;
  __device__ __forceinline__ static void widen(uint4 v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 narrow(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// acc = x_0; acc += x_r for r = 1..n-1, each an fp32 add rounded to nearest
// (written with __fadd_rn so that no contraction or reassociation can occur).
template <int DT, int W>
__device__ __forceinline__ void rank_sum(const uint4 (&raw)[W], int n, float (&acc)[Pack<DT>::kN]) {
  Pack<DT>::widen(raw[0], acc);
#pragma unroll
  for (int r = 1; r < W; r++) {
    if (r < n) {
      float t[Pack<DT>::kN];
      Pack<DT>::widen(raw[r], t);
#pragma unroll
      for (int e = 0; e < Pack<DT>::kN; e++) acc[e] = __fadd_rn(acc[e], t[e]);
    }
  }
}

// ---------------------------------------------------------------------------
// mbarriers, thread-block clusters and distributed shared memory (the fused
// kernels' row statistic and the pipeline's ring).  Every wait built on these
// is bounded by kWaitLimitNs of %globaltimer.
// ---------------------------------------------------------------------------
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Cluster-scope acquire, for the barrier that peers arrive on remotely.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Address of the same shared-memory object in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
// Store a float into a cluster peer's shared memory and count its 4 bytes on
// the peer's mbarrier (asynchronous proxy: no fence over this thread's
// earlier global stores is needed).
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr), "f"(v),
               "r"(bar)
               : "memory");
}
// The same for two 32-bit words (8 bytes, `addr` 8-byte aligned).
__device__ __forceinline__ void st_async_v2_b32(uint32_t addr, uint32_t x, uint32_t y, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "r"(x), "r"(y), "r"(bar)
               : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_barrier, for work in between (every thread of
// every CTA of the cluster, warp-converged; one wait per arrive).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait, with cluster-scope acquire, for the phase of `bar` with the given
// parity; false when it has not completed within limit_ns.
__device__ __forceinline__ bool wait_cluster_phase(uint64_t* bar, uint32_t parity,
                                                   unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1; i < (1u << 30); i++) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
  return false;
}

// Spin for about `ns` nanoseconds of %globaltimer (bounded by an iteration
// count as well).
__device__ __forceinline__ void spin_ns(unsigned long long ns) {
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 0; i < (1u << 30); i++) {
    if (globaltimer() - t0 >= ns) return;
    __nanosleep(256);
  }
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel waits for the grids it depends
// on before its first global memory access (so it is correct after any
// producer), then lets the next PDL-launched kernel of the stream begin its
// launch and prologue while this grid still runs.  Grids here never exceed
// the resident CTA count, so the early trigger cannot keep this grid's own
// CTAs from being scheduled.
// ---------------------------------------------------------------------------
// Ask L2 (not L1) for `bytes` bytes at `p`: 16-byte aligned, a multiple of 16
// bytes.  L2 is coherent for the whole GPU, so this may run before
// griddepcontrol.wait: a load after the wait still sees every write the grid
// it waits for makes, and only the HBM latency moves ahead of the wait.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The same for the 128-byte line that holds `p`, from one thread.
__device__ __forceinline__ void prefetch_line_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

__device__ __forceinline__ void pdl_wait_and_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialisation (and an optional cluster).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                       unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  n++;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    n++;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Stale-line record of a decode: two counts and the first kStaleCap pairs of
// the last call.  Call number c counts in n[c & 1] and, once it may touch
// memory, zeroes n[(c + 1) & 1] for the next call (which waits for this grid
// before logging), so no separate reset has to be queued between calls.
constexpr uint32_t kStaleCap = 65536u;  // == CAR_STALE_LIST_MAX
struct StaleLog {
  unsigned long long n[2];
  uint32_t entry[kStaleCap][2];
};

__device__ __forceinline__ void log_stale(StaleLog* log, int slot, uint32_t rank, uint32_t line) {
  const unsigned long long i = atomicAdd(&log->n[slot], 1ull);
  if (i < kStaleCap) {
    log->entry[i][0] = rank;
    log->entry[i][1] = line;
  }
}

__device__ __forceinline__ void prepare_next_log(StaleLog* log, int slot) {
  if (blockIdx.x == 0 && threadIdx.x == 0) log->n[slot ^ 1] = 0ull;
}

}  // namespace car
