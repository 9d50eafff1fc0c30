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

// Bytes [s, s + 16) of the 32-byte concatenation (a, b), for 0 <= s < 16:
// word selection by s / 4, then a funnel shift by the remaining bytes.
__device__ __forceinline__ uint32_t pick4(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, int q) {
  return q == 0 ? w0 : (q == 1 ? w1 : (q == 2 ? w2 : w3));
}
__device__ __forceinline__ uint4 bytes_at(uint4 a, uint4 b, int s) {
  const int q = s >> 2;
  const uint32_t sh = (uint32_t)(s & 3) * 8u;
  const uint32_t w0 = pick4(a.x, a.y, a.z, a.w, q);
  const uint32_t w1 = pick4(a.y, a.z, a.w, b.x, q);
  const uint32_t w2 = pick4(a.z, a.w, b.x, b.y, q);
  const uint32_t w3 = pick4(a.w, b.x, b.y, b.z, q);
  const uint32_t w4 = pick4(b.x, b.y, b.z, b.w, q);
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh), __funnelshift_r(w2, w3, sh),
                    __funnelshift_r(w3, w4, sh));
}
__device__ __forceinline__ uint4 shfl_down16(uint4 v, int by, int width) {
  return make_uint4(__shfl_down_sync(0xFFFFFFFFu, v.x, by, width), __shfl_down_sync(0xFFFFFFFFu, v.y, by, width),
                    __shfl_down_sync(0xFFFFFFFFu, v.z, by, width), __shfl_down_sync(0xFFFFFFFFu, v.w, by, width));
}
// Evict-first 16-byte store (st.global.cs): the line is not expected to be
// read again soon from L2.
__device__ __forceinline__ void st16_evict_first(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// Aligned rank data whose wire is at least this large per rank is encoded
// by the streaming instance (see ll128_encode_kernel).
constexpr int64_t kStreamWireBytes = 32ll << 20;
__device__ __forceinline__ uint4 shfl_idx16(uint4 v, int src) {
  return make_uint4(__shfl_sync(0xFFFFFFFFu, v.x, src), __shfl_sync(0xFFFFFFFFu, v.y, src),
                    __shfl_sync(0xFFFFFFFFu, v.z, src), __shfl_sync(0xFFFFFFFFu, v.w, src));
}

// Lane c of a half-warp holds data vector c (c < 15) of the line pair.  Wire
// chunk c of the pair is:
//   c <= 6      : data words 2c, 2c+1          -> (x_c, y_c)
//   c == 7      : data word 14, flag            -> (x_7, flag)
//   8 <= c < 15 : data words 2c-1, 2c           -> (y_{c-1}, x_c)
//   c == 15     : data word 29, flag            -> (y_14, flag)
//
// Misaligned data (kMis: the data pointer is element- but not 16-byte
// aligned; P2 "LL128 对齐为何重要" stages such buffers through shared memory):
// lane c loads the aligned 16-byte block c of the pair's range -- every block
// that holds a data byte lies in the same page as that byte, so the load is
// safe -- and rebuilds data vector c from blocks c and c + 1 (one lane
// shuffle and a funnel shift), staying in registers.
template <bool kMis, bool kStream>
__global__ void __launch_bounds__(kWireThreads)
    ll128_encode_kernel(const uint8_t* __restrict__ data, const int64_t data_bytes,
                        const int64_t lines, const uint64_t flag, uint8_t* __restrict__ wire) {
  const int lane = threadIdx.x & 31, c = lane & 15;
  const int64_t pairs = (lines + 1) / 2;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // While the previous grid of the stream finishes: the data of this warp's
  // first line pairs into L2, one request per 128 bytes (lanes 0 and 8 of each
  // half-warp).  8 MiB per rank: 4.04 -> 3.71 us.
  {
    const int64_t p = 2 * (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) + (lane >> 4);
    const int64_t doff = p * 240 + 16 * c;
    if (p < pairs && (c & 7) == 0 && doff < data_bytes) prefetch_line_l2(data + doff);
  }
  pdl_wait_and_release();
  // The streaming instance (kStream: aligned data, a wire of at least
  // kStreamWireBytes per rank, so that a few ranks' wires overflow L2 anyway)
  // keeps the loads of two warp iterations (warp pairs wp and wp + nwarps) in
  // flight per lane before it shuffles and stores them, and writes the wire
  // with evict-first stores.  Measured on GB300 at 128 MiB per rank (graph
  // replay, data rotating above 2x L2): 46.8 us with one load in flight and
  // plain stores, 45.7 us with two loads, 44.8 us with two loads and
  // evict-first stores, 53.8 us with four loads.  The same change made an
  // L2-resident 1 MiB encode 9 % slower (its wire is read from L2 by the next
  // decode) and the misaligned instance 16-47 % slower, so they keep one
  // iteration and plain stores.
  constexpr int kEncodeUnroll = kStream ? 2 : 1;
  for (int64_t wp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; 2 * wp0 < pairs;
       wp0 += kEncodeUnroll * nwarps) {
    uint4 d[kEncodeUnroll];
#pragma unroll
    for (int u = 0; u < kEncodeUnroll; u++) {
      const int64_t p = 2 * (wp0 + u * nwarps) + (lane >> 4);
      d[u] = make_uint4(0u, 0u, 0u, 0u);
      const int64_t doff = p * 240 + 16 * c;
      if (!kMis) {
        if (p < pairs && c < 15 && doff < data_bytes) d[u] = ld_stream(data + doff);
      } else {
        const int m = (int)(reinterpret_cast<uintptr_t>(data) & 15u);
        uint4 blk = make_uint4(0u, 0u, 0u, 0u);
        if (p < pairs && doff - m < data_bytes) blk = ld_stream(data - m + doff);
        const uint4 nxt = shfl_down16(blk, 1, 16);
        if (p < pairs && c < 15 && doff < data_bytes) d[u] = bytes_at(blk, nxt, m);
      }
    }
#pragma unroll
    for (int u = 0; u < kEncodeUnroll; u++) {
      const int64_t p = 2 * (wp0 + u * nwarps) + (lane >> 4);
      const uint64_t x = lo64(d[u]), y = hi64(d[u]);
      const uint64_t y_prev = __shfl_up_sync(kFull, y, 1, 16);
      const uint64_t first = c <= 7 ? x : y_prev;
      const uint64_t second = c <= 6 ? y : ((c == 7 || c == 15) ? flag : x);
      const int64_t line = 2 * p + (c >> 3);
      if (p < pairs && line < lines) {
        if (kStream)
          st16_evict_first(wire + p * 256 + 16 * c, make16(first, second));
        else
          st16(wire + p * 256 + 16 * c, make16(first, second));
      }
    }
  }
}

// Inverse mapping: output vector o (o < 15) of the pair is
//   o <= 6 : (x_o, y_o);  o == 7 : (x_7, x_8);  o >= 8 : (y_o, x_{o+1})
// where (x_c, y_c) is wire chunk c after the rank sum.
//
// Misaligned output (kMisOut): a warp owns the 480 data bytes of its two
// pairs.  Lane b builds aligned output block b (0..30) from data vectors b-1
// and b; the blocks inside the warp's range are stored whole, the first and
// last (shared with the neighbouring warps) and any block past the end of the
// data are stored 2 bytes at a time, only over the bytes this warp owns.
// Allocation-free calls (kPublish): the log is one array that every call on
// the device shares, with n[0] the stale count and n[1] a count of finished
// CTAs.  The last CTA to finish copies the count and the first `cap` pairs
// into the caller's report (uint64 count, 8 reserved bytes, uint32 pairs)
// and clears both counts for the next call, which waits for this grid before
// it logs.  So a call is one kernel: no memset before it and no copy after it
// that would keep programmatic dependent launch from overlapping its
// neighbours.
__device__ __forceinline__ void publish_report(StaleLog* log, uint8_t* report, uint32_t cap) {
  __shared__ unsigned int s_last;
  __threadfence();  // this thread's stale entries are visible to the whole GPU
  __syncthreads();  // ... for every thread of the CTA
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long done = atomicAdd(&log->n[1], 1ull);
    s_last = done == (unsigned long long)gridDim.x - 1ull ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const unsigned long long count = *reinterpret_cast<volatile unsigned long long*>(&log->n[0]);
  const uint32_t listed = count < (unsigned long long)cap ? (uint32_t)count : cap;
  unsigned long long* dst = reinterpret_cast<unsigned long long*>(report);
  if (threadIdx.x == 0) {
    dst[0] = count;
    dst[1] = 0ull;
  }
  const volatile unsigned long long* pairs = reinterpret_cast<const volatile unsigned long long*>(&log->entry[0][0]);
  for (uint32_t i = threadIdx.x; i < listed; i += blockDim.x) dst[2 + i] = pairs[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    log->n[0] = 0ull;
    log->n[1] = 0ull;
  }
}

template <int DT, int W, bool kMisOut, bool kPublish>
__global__ void __launch_bounds__(kWireThreads)
    ll128_decode_reduce_kernel(const RankPtrs wires, const int nranks, const int64_t data_bytes,
                               const int64_t lines, const uint64_t expected, const int max_polls,
                               uint8_t* __restrict__ out, StaleLog* __restrict__ log, const int slot,
                               uint8_t* __restrict__ report, const uint32_t cap) {
  constexpr int R = W > 0 ? W : kMaxRanks;
  const int n = W > 0 ? W : nranks;
  const int lane = threadIdx.x & 31, c = lane & 15;
  const bool flag_lane = (c & 7) == 7;
  const int flag_src = lane | 7;
  const int64_t pairs = (lines + 1) / 2;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // While the previous grid of the stream finishes: the lines of this warp's
  // first pair of line pairs, every rank, into L2 (one request per line, from
  // its first lane).  Measured in graph replay over cold wires: W = 16 at
  // 4 MiB per rank 13.3 -> 12.4 us, W = 8 at 8 MiB 13.6 -> 13.2 us, at
  // 64 MiB 99.9 -> 99.1 us.
  {
    const int64_t p = 2 * (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) + (lane >> 4);
    if (p < pairs && 2 * p + (c >> 3) < lines && (c & 7) == 0) {
#pragma unroll
      for (int r = 0; r < R; r++)
        if (r < n) prefetch_line_l2(static_cast<const uint8_t*>(wires.p[r]) + p * 256 + 16 * c);
    }
  }
  pdl_wait_and_release();
  if (!kPublish) prepare_next_log(log, slot);
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
    if (!kMisOut) {
      if (p < pairs && c < 15 && ooff < data_bytes) st16(out + ooff, make16(first, second));
    } else {
      // data vector d (0..29) of the warp sits in lane d (d < 15) or d + 1
      const int m = (int)(reinterpret_cast<uintptr_t>(out) & 15u);
      const uint4 dv = make16(first, second);
      const int b = lane;
      const int prev = b == 0 ? 0 : (b - 1 < 15 ? b - 1 : b);
      const int cur = b < 15 ? b : (b < 31 ? b + 1 : 31);
      const uint4 va = shfl_idx16(dv, prev);
      const uint4 vb = shfl_idx16(dv, cur);
      const uint4 blk = bytes_at(va, vb, 16 - m);
      const int64_t wbase = 480 * wp;
      const int64_t dw = data_bytes - wbase < 480 ? data_bytes - wbase : 480;
      const int lo = m - 16 * b > 0 ? m - 16 * b : 0;
      const int64_t hi64v = dw - 16 * b + m;
      const int hi = hi64v < 16 ? (int)hi64v : 16;
      uint8_t* dst = out - m + wbase + 16 * b;
      if (b < 31 && lo < hi) {
        if (lo == 0 && hi == 16) {
          st16(dst, blk);
        } else {
          const uint32_t w4[4] = {blk.x, blk.y, blk.z, blk.w};
#pragma unroll
          for (int i = 0; i < 8; i++)
            if (2 * i >= lo && 2 * i < hi)
              *reinterpret_cast<uint16_t*>(dst + 2 * i) = (uint16_t)(w4[i >> 1] >> (16 * (i & 1)));
        }
      }
    }
  }
  if (kPublish) publish_report(log, report, cap);
}

using DecodeFn = void (*)(const RankPtrs, const int, const int64_t, const int64_t, const uint64_t,
                          const int, uint8_t*, StaleLog*, const int, uint8_t*, const uint32_t);

template <int DT, bool kMis, bool kPub>
DecodeFn pick_dt(int W) {
  switch (W) {
    case 2: return ll128_decode_reduce_kernel<DT, 2, kMis, kPub>;
    case 4: return ll128_decode_reduce_kernel<DT, 4, kMis, kPub>;
    case 8: return ll128_decode_reduce_kernel<DT, 8, kMis, kPub>;
    case 16: return ll128_decode_reduce_kernel<DT, 16, kMis, kPub>;
    default: return ll128_decode_reduce_kernel<DT, 0, kMis, kPub>;
  }
}

template <int DT>
DecodeFn pick_dt(int W, bool mis, bool publish) {
  if (publish) return mis ? pick_dt<DT, true, true>(W) : pick_dt<DT, false, true>(W);
  return mis ? pick_dt<DT, true, false>(W) : pick_dt<DT, false, false>(W);
}

DecodeFn pick_decode(int dtype, int W, bool mis, bool publish) {
  switch (dtype) {
    case kBF16: return pick_dt<kBF16>(W, mis, publish);
    case kFP16: return pick_dt<kFP16>(W, mis, publish);
    default: return pick_dt<kFP32>(W, mis, publish);
  }
}

using EncodeFn = void (*)(const uint8_t*, const int64_t, const int64_t, const uint64_t, uint8_t*);

EncodeFn pick_encode(bool mis, int64_t lines) {
  if (mis) return ll128_encode_kernel<true, false>;
  return 128 * lines >= kStreamWireBytes ? ll128_encode_kernel<false, true> : ll128_encode_kernel<false, false>;
}

}  // namespace

cudaError_t ll128_occupancy(int dtype, int W, bool mis, int64_t lines, int* decode_blocks_per_sm,
                            int* encode_blocks_per_sm, bool publish) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      decode_blocks_per_sm, reinterpret_cast<const void*>(pick_decode(dtype, W, mis, publish)), kWireThreads, 0);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      encode_blocks_per_sm,
      reinterpret_cast<const void*>(pick_encode(mis, lines)), kWireThreads, 0);
}

cudaError_t launch_ll128_encode(const void* data, int64_t data_bytes, int64_t lines, uint64_t flag,
                                void* wire, int grid, cudaStream_t s) {
  const bool mis = (reinterpret_cast<uintptr_t>(data) & 15u) != 0;
  return launch_pdl(pick_encode(mis, lines), (unsigned)grid, kWireThreads, 0,
                    s, 1, static_cast<const uint8_t*>(data), data_bytes, lines, flag, static_cast<uint8_t*>(wire));
}

cudaError_t launch_ll128_decode_reduce(int dtype, int W, const RankPtrs& wires, int64_t data_bytes,
                                       int64_t lines, uint64_t expected, int max_polls, void* out,
                                       StaleLog* log, int slot, int grid, cudaStream_t s, void* report,
                                       uint32_t cap) {
  const bool mis = (reinterpret_cast<uintptr_t>(out) & 15u) != 0;
  return launch_pdl(pick_decode(dtype, W, mis, report != nullptr), (unsigned)grid, kWireThreads, 0, s, 1, wires, W,
                    data_bytes, lines, expected, max_polls, static_cast<uint8_t*>(out), log, slot,
                    static_cast<uint8_t*>(report), cap);
}

}  // namespace car
