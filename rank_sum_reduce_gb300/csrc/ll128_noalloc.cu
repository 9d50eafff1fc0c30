// ll128_noalloc.cu -- LL128 validate + decode + rank-sum reduce for callers
// that must not allocate device memory.
//
// Who needs this: car_create() calls cudaMalloc for the handle's stale-line
// log.  Some callers cannot do that: code running inside an allocator's own
// callbacks (re-entering the allocator would deadlock), processes where a
// framework's caching pool already holds all free device memory (a fresh
// cudaMalloc fails), and latency-critical paths that cannot afford the device
// synchronisation cudaMalloc/cudaFree can imply.  This entry point needs no
// handle: its stale-line log lives in a fixed device array that the library
// itself carries (the array below), so no call allocates.
//
// The array is process-wide and per device: every call on a device shares it.
// Each call is a single kernel whose last CTA to finish copies the report to
// the caller's buffer and clears the array's two counts for the next call;
// the stale pairs themselves stay until the next call overwrites them.  Calls
// that overlap on the GPU (for example on two streams at once) race on it and
// corrupt each other's report.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "../../include/car.h"
#include "car_device.cuh"
#include "car_launch.h"

namespace car {
namespace {

// The stale-line log of this entry point, laid out as StaleLog: the stale
// count, a count of finished CTAs, then up to kStaleCap (rank, line) pairs.
// Zero when the library is loaded, and cleared again by every call.
constexpr size_t kScratchWords = sizeof(StaleLog) / sizeof(unsigned long long);
static_assert(sizeof(StaleLog) % sizeof(unsigned long long) == 0, "StaleLog size");
static __device__ __align__(256) unsigned long long g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready;
  StaleLog* log;          // device address of g_noalloc_scratch on this device
  int num_sms;
  int per_sm[3][5][2];    // decode blocks per SM by dtype, W instance and output alignment
                          // (the aligned or the misaligned-output kernel; 0 = not asked yet)
};
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

car_status cuda_error(cudaError_t e, const char* where) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  set_last_error(msg);
  return CAR_ERR_CUDA;
}

int w_instance(int W) {
  switch (W) {
    case 2: return 1;
    case 4: return 2;
    case 8: return 3;
    case 16: return 4;
    default: return 0;
  }
}

// Once per device, with that device current: look up where the array lives
// on the device (the host-side name is only a stand-in for it) and read the
// SM count.  The first call on each device runs this, and the address is
// kept for the life of the process (a device reset after that first call is
// not supported: it could move the array).
car_status setup(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) {
    set_last_error("car_ll128_decode_reduce_noalloc: device index beyond 63");
    return CAR_ERR_ARG;
  }
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(noalloc scratch)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_error(e, "SM count");
    st.log = static_cast<StaleLog*>(ptr);
    st.num_sms = sms;
    st.ready = true;
  }
  *out = &st;
  return CAR_OK;
}

}  // namespace
}  // namespace car

extern "C" car_status car_ll128_decode_reduce_noalloc(int W, int64_t M, int64_t N, car_dtype dtype,
                                                     const void* const* wires, uint64_t expected_flag,
                                                     int max_polls, void* ar_out, void* stale_out,
                                                     uint32_t cap, void* stream) {
  using namespace car;
  if (W < 1 || W > kMaxRanks || M < 1 || N < 1 || max_polls < 1) return CAR_ERR_ARG;
  if (dtype != CAR_BF16 && dtype != CAR_FP16 && dtype != CAR_FP32) return CAR_ERR_ARG;
  if (cap > kStaleCap) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "car_ll128_decode_reduce_noalloc: cap %u exceeds the fixed stale list of %u entries", cap,
             kStaleCap);
    set_last_error(msg);
    return CAR_ERR_SIZE;
  }
  const int es = dtype == CAR_FP32 ? 4 : 2;
  if (N > (int64_t)INT32_MAX / es || (N * es) % 16 != 0) return CAR_ERR_SIZE;
  if (M > ((int64_t)1 << 56) / (N * es)) return CAR_ERR_SIZE;
  const int64_t D = M * N * es;
  const int64_t lines = (D + 119) / 120;
  if (lines > (int64_t)UINT32_MAX) return CAR_ERR_SIZE;
  if (!wires || !ar_out || !stale_out) return CAR_ERR_ARG;
  RankPtrs tbl = {};
  for (int r = 0; r < W; r++) {
    if (!wires[r]) return CAR_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(wires[r]) & 15u) return CAR_ERR_ALIGN;
    tbl.p[r] = wires[r];
  }
  if ((reinterpret_cast<uintptr_t>(ar_out) % (uintptr_t)es) || (reinterpret_cast<uintptr_t>(stale_out) & 15u))
    return CAR_ERR_ALIGN;

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  DeviceState* st = nullptr;
  int grid = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    car_status s = setup(dev, &st);
    if (s != CAR_OK) return s;
    const bool mis = (reinterpret_cast<uintptr_t>(ar_out) & 15u) != 0;  // the instance launched below
    int& per_sm = st->per_sm[dtype][w_instance(W)][mis ? 1 : 0];
    if (per_sm == 0) {
      int enc = 0;
      e = ll128_occupancy(dtype, W, mis, lines, &per_sm, &enc, true);
      if (e != cudaSuccess) {
        per_sm = 0;
        return cuda_error(e, "ll128 occupancy");
      }
      per_sm = std::max(per_sm, 1);
    }
    const int64_t pairs = (lines + 1) / 2;
    const int64_t blocks = ((pairs + 1) / 2 + kWireThreads / 32 - 1) / (kWireThreads / 32);
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)per_sm * st->num_sms));
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // One kernel: its last CTA writes the report and clears the array for the
  // next call (see publish_report in ll128.cu).
  e = launch_ll128_decode_reduce(dtype, W, tbl, D, lines, expected_flag, max_polls, ar_out, st->log, 0, grid, s,
                                 stale_out, cap);
  if (e != cudaSuccess) return cuda_error(e, "ll128_decode_reduce launch (noalloc)");
  return CAR_OK;
}
