// ll128.cu -- LL128 line encode, and validate + decode + rank-sum reduce.
//
// P2 "NCCL 专家课程 14：Simple、LL、LL128 的线格式、同步与真实性能边界",
// sections "LL128 的 128-byte line" (128-byte line = 15 data words + 1 flag
// word, 8 lanes x 16 bytes cover a line, the lane with tid % 8 == 7 carries
// the flag in its second word) and "LL128 的 warp-level ready 检查" (flag
// lanes compare, the warp votes, data is used once the flag matches; a sender
// writes its data words with the flag in the flag lane's second word).
//
// GB300 design: a 16-lane half-warp owns a pair of consecutive lines (256 wire
// bytes = 240 data bytes = 15 whole 16-byte output vectors), so every wire
// read and every output write is a full, aligned 16-byte access and a warp
// touches 512 contiguous wire bytes per rank.  The 120-byte data pieces are
// re-aligned with one 64-bit lane shuffle instead of a trip through shared
// memory.  The flag check happens on the same read as the data (one pass over
// HBM); a stale line is re-read only when max_polls > 1, at most max_polls - 1
// times.  Roofline: HBM, W * 128 wire bytes read + 120 bytes written per line.
#include "car_device.cuh"
#include "car_launch.h"

namespace car {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Lane c of a half-warp holds data vector c (c < 15) of the line pair.  Wire
// chunk c of the pair is:
//   c <= 6      : data words 2c, 2c+1          -> (x_c, y_c)
//   c == 7      : data word 14, flag            -> (x_7, flag)
//   8 <= c < 15 : data words 2c-1, 2c           -> (y_{c-1}, x_c)
//   c == 15     : data word 29, flag            -> (y_14, flag)
__global__ void __launch_bounds__(kWireThreads)
    ll128_encode_kernel(const uint8_t* __restrict__ data, const int64_t data_bytes,
                        const int64_t lines, const uint64_t flag, uint8_t* __restrict__ wire) {
  const int lane = threadIdx.x & 31, c = lane & 15;
  const int64_t pairs = (lines + 1) / 2;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  pdl_wait_and_release();
  for (int64_t wp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; 2 * wp < pairs;
       wp += nwarps) {
    const int64_t p = 2 * wp + (lane >> 4);
    uint4 d = make_uint4(0u, 0u, 0u, 0u);
    const int64_t doff = p * 240 + 16 * c;
    if (p < pairs && c < 15 && doff < data_bytes) d = ld_stream(data + doff);
    const uint64_t x = lo64(d), y = hi64(d);
    const uint64_t y_prev = __shfl_up_sync(kFull, y, 1, 16);
    const uint64_t first = c <= 7 ? x : y_prev;
    const uint64_t second = c <= 6 ? y : ((c == 7 || c == 15) ? flag : x);
    const int64_t line = 2 * p + (c >> 3);
    if (p < pairs && line < lines) st16(wire + p * 256 + 16 * c, make16(first, second));
  }
}

// Inverse mapping: output vector o (o < 15) of the pair is
//   o <= 6 : (x_o, y_o);  o == 7 : (x_7, x_8);  o >= 8 : (y_o, x_{o+1})
// where (x_c, y_c) is wire chunk c after the rank sum.
template <int DT, int W>
__global__ void __launch_bounds__(kWireThreads)
    ll128_decode_reduce_kernel(const RankPtrs wires, const int nranks, const int64_t data_bytes,
                               const int64_t lines, const uint64_t expected, const int max_polls,
                               uint8_t* __restrict__ out, StaleLog* __restrict__ log, const int slot) {
  constexpr int R = W > 0 ? W : kMaxRanks;
  const int n = W > 0 ? W : nranks;
  const int lane = threadIdx.x & 31, c = lane & 15;
  const bool flag_lane = (c & 7) == 7;
  const int flag_src = lane | 7;
  const int64_t pairs = (lines + 1) / 2;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  pdl_wait_and_release();
  prepare_next_log(log, slot);
  for (int64_t wp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; 2 * wp < pairs;
       wp += nwarps) {
    const int64_t p = 2 * wp + (lane >> 4);
    const int64_t line = 2 * p + (c >> 3);
    const bool live = p < pairs && line < lines;
    const int64_t woff = p * 256 + 16 * c;

    uint4 raw[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
      if (r < n) {
        raw[r] = make_uint4(0u, 0u, 0u, 0u);
        if (live) raw[r] = ld_wire(static_cast<const uint8_t*>(wires.p[r]) + woff);
      }
    }
    uint32_t bad = 0;
    if (live && flag_lane) {
#pragma unroll
      for (int r = 0; r < R; r++)
        if (r < n && hi64(raw[r]) != expected) bad |= 1u << r;
    }
    // bounded re-polls: lines of a stale group re-read all their chunks
    for (int poll = 1; poll < max_polls; poll++) {
      const uint32_t group_bad = __shfl_sync(kFull, bad, flag_src);
      if (!__any_sync(kFull, group_bad != 0)) break;
      if (group_bad) {
#pragma unroll
        for (int r = 0; r < R; r++)
          if (r < n) raw[r] = ld_wire_poll(static_cast<const uint8_t*>(wires.p[r]) + woff);
        if (flag_lane) {
          bad = 0;
#pragma unroll
          for (int r = 0; r < R; r++)
            if (r < n && hi64(raw[r]) != expected) bad |= 1u << r;
        }
      }
    }
    const uint32_t group_bad = __shfl_sync(kFull, bad, flag_src);
    if (bad) {
      for (int r = 0; r < n; r++)
        if (bad >> r & 1u) log_stale(log, slot, (uint32_t)r, (uint32_t)line);
    }

    uint4 sum = make_uint4(0u, 0u, 0u, 0u);
    if (!group_bad) {
      float acc[Pack<DT>::kN];
      rank_sum<DT, R>(raw, n, acc);
      sum = Pack<DT>::narrow(acc);
    }
    const uint64_t x = lo64(sum), y = hi64(sum);
    const uint64_t x_next = __shfl_down_sync(kFull, x, 1, 16);
    const uint64_t first = c <= 7 ? x : y;
    const uint64_t second = c <= 6 ? y : x_next;
    const int64_t ooff = p * 240 + 16 * c;
    if (p < pairs && c < 15 && ooff < data_bytes) st16(out + ooff, make16(first, second));
  }
}

using DecodeFn = void (*)(const RankPtrs, const int, const int64_t, const int64_t, const uint64_t,
                          const int, uint8_t*, StaleLog*, const int);

template <int DT>
DecodeFn pick_dt(int W) {
  switch (W) {
    case 2: return ll128_decode_reduce_kernel<DT, 2>;
    case 4: return ll128_decode_reduce_kernel<DT, 4>;
    case 8: return ll128_decode_reduce_kernel<DT, 8>;
    case 16: return ll128_decode_reduce_kernel<DT, 16>;
    default: return ll128_decode_reduce_kernel<DT, 0>;
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

cudaError_t ll128_occupancy(int dtype, int W, int* decode_blocks_per_sm, int* encode_blocks_per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      decode_blocks_per_sm, reinterpret_cast<const void*>(pick_decode(dtype, W)), kWireThreads, 0);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      encode_blocks_per_sm, reinterpret_cast<const void*>(ll128_encode_kernel), kWireThreads, 0);
}

cudaError_t launch_ll128_encode(const void* data, int64_t data_bytes, int64_t lines, uint64_t flag,
                                void* wire, int grid, cudaStream_t s) {
  return launch_pdl(ll128_encode_kernel, (unsigned)grid, kWireThreads, 0, s, 1, static_cast<const uint8_t*>(data),
                    data_bytes, lines, flag, static_cast<uint8_t*>(wire));
}

cudaError_t launch_ll128_decode_reduce(int dtype, int W, const RankPtrs& wires, int64_t data_bytes,
                                       int64_t lines, uint64_t expected, int max_polls, void* out,
                                       StaleLog* log, int slot, int grid, cudaStream_t s) {
  return launch_pdl(pick_decode(dtype, W), (unsigned)grid, kWireThreads, 0, s, 1, wires, W, data_bytes, lines,
                    expected, max_polls, static_cast<uint8_t*>(out), log, slot);
}

}  // namespace car
