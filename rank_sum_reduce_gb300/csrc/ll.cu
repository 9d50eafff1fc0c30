// ll.cu -- LL line encode, and validate + decode + rank-sum reduce.
//
// P2 "NCCL 专家课程 14：Simple、LL、LL128 的线格式、同步与真实性能边界",
// sections "LL 的 16-byte FIFO line" (a 16-byte line is {data1, flag1, data2,
// flag2}, flags after their data) and "LL 如何发布和等待 flag" (the sender
// writes the whole line in one 16-byte store; the receiver reads the line with
// one 16-byte load, accepts it when both flags equal the expected flag, and
// decodes data1 + (data2 << 32)).
//
// GB300 design: encode turns each 16-byte data vector into two lines, a warp
// writing 512 contiguous wire bytes per store; decode gives one line per thread per rank, so
// every access is a full 16-byte load and a warp stores 256 contiguous output
// bytes.  Roofline: HBM, W * 16 wire bytes read + 8 bytes written per line.
#include "car_device.cuh"
#include "car_launch.h"

namespace car {
namespace {

// A warp takes 32 consecutive data vectors (lane t loads vector t) and writes
// their 64 lines with two stores, each over 512 contiguous wire bytes: in
// store k, lane t writes line 32k + t, the low (t even) or high (t odd) data
// word of vector 16k + t/2, fetched from its lane by shuffle.  Storing the two
// lines of a thread's own vector instead (two stores 16 bytes apart, each
// warp store spread over 1024 bytes) measured 0.75 against 0.86 of the copy
// peak at 64 MiB.
__global__ void __launch_bounds__(kWireThreads)
    ll_encode_kernel(const uint4* __restrict__ data, const int64_t nvec, const uint32_t flag,
                     uint4* __restrict__ wire) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // While the previous grid of the stream finishes: this warp's first 32
  // data vectors into L2, one request per 128 bytes (64 MiB: 34.8 -> 32.8 us).
  {
    const int64_t i = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 32 + lane;
    if (i < nvec && (lane & 7) == 0) prefetch_line_l2(data + i);
  }
  pdl_wait_and_release();
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w * 32 < nvec; w += nwarps) {
    const int64_t i = w * 32 + lane;
    const uint4 d = i < nvec ? ld_stream(data + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < 2; k++) {
      const int src = 16 * k + (lane >> 1);
      const uint32_t x = __shfl_sync(0xFFFFFFFFu, d.x, src), y = __shfl_sync(0xFFFFFFFFu, d.y, src);
      const uint32_t z = __shfl_sync(0xFFFFFFFFu, d.z, src), u = __shfl_sync(0xFFFFFFFFu, d.w, src);
      const int64_t line = 64 * w + 32 * k + lane;  // = data word index
      if (line < 2 * nvec) st16(wire + line, (lane & 1) ? make_uint4(z, flag, u, flag) : make_uint4(x, flag, y, flag));
    }
  }
}

template <int DT, int W>
__global__ void __launch_bounds__(kWireThreads)
    ll_decode_reduce_kernel(const RankPtrs wires, const int nranks, const int64_t lines,
                            const uint32_t expected, const int max_polls, uint2* __restrict__ out,
                            StaleLog* __restrict__ log, const int slot) {
  constexpr int R = W > 0 ? W : kMaxRanks;
  const int n = W > 0 ? W : nranks;
  // While the previous grid of the stream finishes: this thread's first line
  // of every rank into L2, one request per 8 lines (128 bytes).  Measured in
  // graph replay over cold wires: W = 8 at 8 MiB per rank 22.3 -> 20.7 us,
  // 64 MiB 172.7 -> 170.9 us; W = 16 at 4 MiB 22.4 -> 22.9 us.  (Equal
  // contiguous shares per CTA, as in the reduce kernels, made this kernel
  // slower at 64 MiB: 197 us.)
  {
    const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (v < lines && (threadIdx.x & 7) == 0) {
#pragma unroll
      for (int r = 0; r < R; r++)
        if (r < n) prefetch_line_l2(static_cast<const uint4*>(wires.p[r]) + v);
    }
  }
  pdl_wait_and_release();
  prepare_next_log(log, slot);
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < lines; i += step) {
    uint4 raw[R];
#pragma unroll
    for (int r = 0; r < R; r++)
      if (r < n) raw[r] = ld_wire(static_cast<const uint4*>(wires.p[r]) + i);
    uint32_t bad = 0;
#pragma unroll
    for (int r = 0; r < R; r++)
      if (r < n && (raw[r].y != expected || raw[r].w != expected)) bad |= 1u << r;
    for (int poll = 1; poll < max_polls && bad; poll++) {
#pragma unroll
      for (int r = 0; r < R; r++)
        if (r < n) raw[r] = ld_wire_poll(static_cast<const uint4*>(wires.p[r]) + i);
      bad = 0;
#pragma unroll
      for (int r = 0; r < R; r++)
        if (r < n && (raw[r].y != expected || raw[r].w != expected)) bad |= 1u << r;
    }
    uint2 o = make_uint2(0u, 0u);
    if (bad) {
      for (int r = 0; r < n; r++)
        if (bad >> r & 1u) log_stale(log, slot, (uint32_t)r, (uint32_t)i);
    } else {
      // decoded data word of rank r: data1 | data2 << 32 = (raw.x, raw.z)
      uint4 words[R];
#pragma unroll
      for (int r = 0; r < R; r++)
        if (r < n) words[r] = make_uint4(raw[r].x, raw[r].z, 0u, 0u);
      float acc[Pack<DT>::kN];
      rank_sum<DT, R>(words, n, acc);
      const uint4 s = Pack<DT>::narrow(acc);
      o = make_uint2(s.x, s.y);
    }
    out[i] = o;
  }
}

using DecodeFn = void (*)(const RankPtrs, const int, const int64_t, const uint32_t, const int,
                          uint2*, StaleLog*, const int);

template <int DT>
DecodeFn pick_dt(int W) {
  switch (W) {
    case 2: return ll_decode_reduce_kernel<DT, 2>;
    case 4: return ll_decode_reduce_kernel<DT, 4>;
    case 8: return ll_decode_reduce_kernel<DT, 8>;
    case 16: return ll_decode_reduce_kernel<DT, 16>;
    default: return ll_decode_reduce_kernel<DT, 0>;
  }
}

DecodeFn pick_decode(int dtype, int W) {
  switch (dtype) {
    case kBF16: return pick_dt<kBF16>(W);
    case kFP16: return pick_dt<kFP16>(W);
    default: return pick_dt<kFP32>(W);
  }
}

}  // namespace

cudaError_t ll_occupancy(int dtype, int W, int* decode_blocks_per_sm, int* encode_blocks_per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      decode_blocks_per_sm, reinterpret_cast<const void*>(pick_decode(dtype, W)), kWireThreads, 0);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      encode_blocks_per_sm, reinterpret_cast<const void*>(ll_encode_kernel), kWireThreads, 0);
}

cudaError_t launch_ll_encode(const void* data, int64_t data_bytes, uint32_t flag, void* wire,
                             int grid, cudaStream_t s) {
  return launch_pdl(ll_encode_kernel, (unsigned)grid, kWireThreads, 0, s, 1, static_cast<const uint4*>(data),
                    data_bytes / 16, flag, static_cast<uint4*>(wire));
}

cudaError_t launch_ll_decode_reduce(int dtype, int W, const RankPtrs& wires, int64_t data_bytes,
                                    uint32_t expected, int max_polls, void* out, StaleLog* log, int slot,
                                    int grid, cudaStream_t s) {
  return launch_pdl(pick_decode(dtype, W), (unsigned)grid, kWireThreads, 0, s, 1, wires, W, data_bytes / 8,
                    expected, max_polls, static_cast<uint2*>(out), log, slot);
}

}  // namespace car
