// api.cu -- the C ABI of libcar (include/car.h): argument checks, handles,
// launch shapes, stale-line reports.  Every operation runs in the kernels of
// reduce.cu, fused.cu, ll128.cu and ll.cu; nothing here computes results.
//
// Argument rules follow the problem statement on the pages:
//   P1 "SGLang Custom AllReduce v1 线程模型和工作原理细节", section
//      "一次调用给 kernel 什么：参数与 grid" (message bytes a multiple of 16;
//      same size and type on every rank) and "线程模型：16 字节一个单位"
//      (16-byte aligned packed units);
//   P3 "0-custom-all-reduce", "调用" (up to 16 ranks) and "5. 写回"
//      (output may alias the input);
//   P2 "NCCL 专家课程 14：Simple、LL、LL128 的线格式、同步与真实性能边界",
//      "LL 如何发布和等待 flag" (waits are bounded: the page's loops check for
//      abort; here a poll count bounds them).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>

#include "../../include/car.h"
#include "car_device.cuh"
#include "car_launch.h"

static_assert(car::kStaleCap == CAR_STALE_LIST_MAX, "stale list capacity mismatch");

struct car_ctx {
  int W;
  int64_t M, N;
  int dtype;
  int es;
  int64_t D;            // bytes per rank
  int64_t nvec;         // 16-byte vectors per rank
  int vec_per_row;      // 16-byte vectors per row
  int device;
  int num_sms;
  int reduce_grid;
  int two_shot_grid;
  bool fused_ok;        // row short enough for the fused kernel
  car::FusedShape fused_auto;
  car::FusedShape fused;
  bool tma_ok;          // row fits the shared-memory ring of the pipelined kernel
  car::FusedTmaShape tma_auto;
  car::FusedTmaShape tma;
  int fused_kernel_auto;  // CAR_FUSED_ROWS or CAR_FUSED_PIPELINE
  int fused_kernel;
  unsigned int* d_err;  // bounded-wait failures reported by kernels (device)
  car::WaitHook hook;   // the fused row kernel's partial-exchange wait limit and test delay
  int64_t ll128_lines;
  int ll128_encode_grid[2], ll128_decode_grid[2];  // [1]: the misaligned instances
  int64_t ll_lines;
  int ll_encode_grid, ll_decode_grid;
  bool lamport_ok;              // bf16 and a row the Lamport receive kernel takes
  car::FusedShape lamport;
  int lamport_grid;             // fill / push kernels
  car::StaleLog* log[3];       // [0] LL128, [1] LL, [2] Lamport (device)
  cudaStream_t last_stream[3];
  bool decoded[3];
  uint64_t calls[3];           // decode calls so far; call c counts in log->n[c & 1]
  int last_slot[3];
};

namespace {

std::mutex g_mu;
std::unordered_set<const car_ctx*> g_live;
thread_local char g_err[256] = "";

car_status cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_err, sizeof(g_err), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  return CAR_ERR_CUDA;
}

bool live(const car_ctx* h) {
  if (!h) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_live.count(h) != 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by every call on a handle: the handle is live and its device
// is the current one.
car_status check_handle(const car_ctx* h) {
  if (!live(h)) return CAR_ERR_HANDLE;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h->device) {
    snprintf(g_err, sizeof(g_err), "handle belongs to device %d, current device is %d", h->device, dev);
    return CAR_ERR_ARG;
  }
  return CAR_OK;
}

car_status check_table(const car_ctx* h, const void* const* ptrs, car::RankPtrs* out) {
  if (!ptrs) return CAR_ERR_ARG;
  std::memset(out, 0, sizeof(*out));
  for (int r = 0; r < h->W; r++) {
    if (!ptrs[r]) return CAR_ERR_ARG;
    if (!aligned16(ptrs[r])) return CAR_ERR_ALIGN;
    out->p[r] = ptrs[r];
  }
  return CAR_OK;
}

car_status check_dev(const void* p) {
  if (!p) return CAR_ERR_ARG;
  return aligned16(p) ? CAR_OK : CAR_ERR_ALIGN;
}

// Rank data of the LL128 calls needs only element alignment.
car_status check_dev_elem(const void* p, int es) {
  if (!p) return CAR_ERR_ARG;
  return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)es) == 0 ? CAR_OK : CAR_ERR_ALIGN;
}

int clamp_grid(int64_t needed, int per_sm, int num_sms) {
  const int64_t cap = (int64_t)std::max(per_sm, 1) * num_sms;
  return (int)std::max<int64_t>(1, std::min(needed, cap));
}

int round_up32(int64_t v) { return (int)((v + 31) / 32 * 32); }

// Automatic shape of a row-split kernel (the fused row kernel and the Lamport
// receive), given which (W, vectors per thread) instances are compiled and
// their thread limits.  A row is split over a cluster of c = 8 or 4 CTAs (the
// largest that qualifies) when
//  * each CTA keeps at least 128 16-byte vectors of the row,
//  * the c * M CTAs stay within 7/8 of the SMs (one wave of clusters), and
//  * there are at most 16 rows, or each row brings at least 48 KB of inputs;
// otherwise one CTA takes a row, with the fewest vectors per thread that the
// compiled instances allow.  A row too wide for one CTA's threads takes the
// smallest cluster whose CTAs cover it.
//
// Measured on GB300 for the fused row kernel, with the partials pushed by
// st.async (graph replay over cold inputs, bf16; us per call, rule's choice
// against one CTA per row): W = 8, N = 8192: M = 1 1.97 / 3.01, M = 32
// (c = 4) 2.70 / 3.19; W = 8, N = 4096, M = 1 (c = 4) 1.90 / 2.19; W = 2,
// N = 8192, M = 32 (c = 4) 2.26 / 2.45.  Where the rule keeps one CTA per row
// it was as fast or faster: W = 4, N = 4096, M = 32: 2.09 against 2.20 with
// four CTAs; W = 2, N = 2048, M = 1: 1.48 against 1.64 with two.
//
// With prefer_half_ctas, a shape that would need a 1024-thread CTA with one
// vector per thread takes 512 threads with two vectors instead when that
// instance exists.  Measured for the fused row kernel (one CTA per row, bf16,
// N = 8192, graph replay over cold inputs, us per call, 512 x 2 against
// 1024 x 1): W = 4, M = 128 3.51 / 3.61; W = 4, M = 64 2.74 / 2.85; W = 2,
// M = 128 2.89 / 3.05.
template <class HasVariant, class MaxThreads>
car::FusedShape row_split_shape(int W, int64_t M, int V, int num_sms, HasVariant has_variant,
                                MaxThreads max_threads, bool prefer_half_ctas) {
  auto fit = [&](int c, car::FusedShape* out) {
    const int chunk = (V + c - 1) / c;
    for (int vpt = 1; vpt <= 2; vpt++) {
      if (!has_variant(W, vpt)) continue;
      const int t = std::max(32, round_up32((chunk + vpt - 1) / vpt));
      if (vpt == 1 && prefer_half_ctas && t > 512 && has_variant(W, 2) &&
          std::max(32, round_up32((chunk + 1) / 2)) <= max_threads(W, 2))
        continue;
      if (t <= max_threads(W, vpt)) {
        *out = car::FusedShape{c, t, vpt, 1};
        return true;
      }
    }
    return false;
  };
  car::FusedShape sh;
  const int64_t row_in = (int64_t)(W + 1) * V * 16;
  for (int c = 8; c >= 4; c /= 2) {
    if (V / c < 128 || (int64_t)c * M > num_sms - num_sms / 8 || (M > 16 && row_in < 48 * 1024)) continue;
    if (fit(c, &sh)) return sh;
  }
  for (int c = 1; c <= 8; c *= 2)
    if (fit(c, &sh)) return sh;
  return car::FusedShape{8, std::max(32, round_up32((V + 7) / 8)), 1, 1};  // rows past CAR_MAX_ROW_BYTES only
}

car::FusedShape auto_fused_shape(int W, int64_t M, int V, int num_sms) {
  return row_split_shape(W, M, V, num_sms, car::fused_has_variant, car::fused_max_threads, true);
}

bool shape_valid(int W, int V, const car::FusedShape& sh) {
  if (sh.cluster != 1 && sh.cluster != 2 && sh.cluster != 4 && sh.cluster != 8) return false;
  if (!car::fused_has_variant(W, sh.vpt)) return false;
  if (sh.threads < 32 || sh.threads % 32 != 0 || sh.threads > car::fused_max_threads(W, sh.vpt)) return false;
  const int64_t chunk = (V + sh.cluster - 1) / sh.cluster;
  return (int64_t)sh.threads * sh.vpt >= chunk;
}

// The pipelined kernel is faster once there are more rows than SMs and a row
// slice (N * s bytes, one bulk copy per rank) is larger than 8 KB.  Measured on
// GB300 against the row kernel (both fetching their first row into L2 before
// the PDL wait), N = 8192 bf16: at M = 152, W = 8 5.8 (rows) against 6.5 us
// (pipeline), W = 2 3.3 against 3.8; at M = 184, W = 8 8.2 against 7.5, W = 2
// 5.3 against 4.5; at M = 456, W = 8 15.4 against 13.4; at M = 1024 28.2
// (pipeline) against 32.3; 12 KB slices, W = 8, M = 1024, N = 6144 bf16: 21.7
// against 25.9; W = 4, M = 1024, N = 3072 fp32: 14.9 against 18.2.  With 8 KB
// slices and smaller the persistent CTA finishes its rows one after another
// (each behind the row statistic's barriers), and the row kernel, many CTAs
// per SM, keeps more rows in flight: W = 4,
// M = 1024, N = 4096 bf16 11.8 (rows) against 13.0 us; W = 8, M = 4096,
// N = 2048 29.2 against 46.1; W = 2, M = 4096, N = 1024 8.9 against 27.4; a
// deeper ring with several issuing lanes did not close the gap.
int auto_fused_kernel(const car_ctx* h) {
  const bool big_slices = h->N * (int64_t)h->es > 8192;
  return (h->tma_ok && big_slices && h->M > (int64_t)h->num_sms) ? CAR_FUSED_PIPELINE : CAR_FUSED_ROWS;
}

// Row-kernel shape for the Lamport receive step: the same rules as the fused
// row kernel, within the Lamport kernel's compiled instances.
car::FusedShape auto_lamport_shape(int W, int64_t M, int V, int num_sms) {
  return row_split_shape(W, M, V, num_sms, car::lamport_has_variant, car::lamport_max_threads, false);
}

car_status finish_fused_shape(car_ctx* h, car::FusedShape sh) {
  int groups = 0;
  cudaError_t e = car::fused_resident_groups(h->dtype, h->W, sh, h->num_sms, &groups);
  if (e != cudaSuccess) return cuda_fail(e, "fused occupancy");
  sh.groups = (int)std::max<int64_t>(1, std::min<int64_t>(h->M, std::max(groups, 1)));
  h->fused = sh;
  return CAR_OK;
}

// The log slot of the next decode of this kind (its kernel zeroes the other).
int next_log_slot(car_ctx* h, int which) {
  const int slot = (int)(h->calls[which] & 1u);
  h->calls[which]++;
  h->last_slot[which] = slot;
  return slot;
}

car_status decode_common(car_ctx* h, int which, const void* const* wires, int max_polls,
                         void* ar_out, cudaStream_t s, car::RankPtrs* tbl) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  if (max_polls < 1) return CAR_ERR_ARG;
  if ((st = check_table(h, wires, tbl)) != CAR_OK) return st;
  // LL128 output may sit at any element offset; LL output stays 16-byte aligned
  if ((st = which == 0 ? check_dev_elem(ar_out, h->es) : check_dev(ar_out)) != CAR_OK) return st;
  h->last_stream[which] = s;
  h->decoded[which] = true;
  return CAR_OK;
}

car_status report_common(car_ctx* h, int which, car_stale_report* out) {
  if (!live(h)) return CAR_ERR_HANDLE;
  if (!out || (out->cap > 0 && !out->entries)) return CAR_ERR_ARG;
  out->n_stale = 0;
  out->n_listed = 0;
  if (!h->decoded[which]) return CAR_OK;
  cudaError_t e = cudaStreamSynchronize(h->last_stream[which]);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned long long n = 0;
  e = cudaMemcpy(&n, &h->log[which]->n[h->last_slot[which]], sizeof(n), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read stale count");
  const uint64_t listed = std::min<uint64_t>(n, std::min<uint64_t>(out->cap, car::kStaleCap));
  if (listed) {
    e = cudaMemcpy(out->entries, h->log[which]->entry, listed * 2 * sizeof(uint32_t),
                   cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read stale list");
  }
  // Clear the count just read.  A decode zeroes only the other slot (for the
  // call after it), so a single decode captured in a CUDA graph would
  // otherwise add every replay's stale lines to the same count.
  if (n) {
    e = cudaMemsetAsync(&h->log[which]->n[h->last_slot[which]], 0, sizeof(n), h->last_stream[which]);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->last_stream[which]);
    if (e != cudaSuccess) return cuda_fail(e, "clear stale count");
  }
  out->n_stale = n;
  out->n_listed = (uint32_t)listed;
  return n ? CAR_ERR_STALE_FLAG : CAR_OK;
}

}  // namespace

namespace car {
void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }
}  // namespace car

extern "C" {

const char* car_status_string(car_status s) {
  switch (s) {
    case CAR_OK: return "CAR_OK";
    case CAR_ERR_ARG: return "CAR_ERR_ARG: invalid argument";
    case CAR_ERR_ALIGN: return "CAR_ERR_ALIGN: device pointer not 16-byte aligned";
    case CAR_ERR_SIZE: return "CAR_ERR_SIZE: unsupported size";
    case CAR_ERR_CUDA: return "CAR_ERR_CUDA: CUDA runtime error";
    case CAR_ERR_STALE_FLAG: return "CAR_ERR_STALE_FLAG: stale lines found";
    case CAR_ERR_HANDLE: return "CAR_ERR_HANDLE: invalid handle";
    case CAR_ERR_TIMEOUT: return "CAR_ERR_TIMEOUT: a kernel gave up a bounded wait";
  }
  return "unknown car_status";
}

const char* car_last_error(void) { return g_err; }

car_status car_create(int W, int64_t M, int64_t N, car_dtype dtype, car_ctx** out) {
  if (!out) return CAR_ERR_ARG;
  *out = nullptr;
  g_err[0] = 0;
  if (W < 1 || W > car::kMaxRanks || M < 1 || N < 1) return CAR_ERR_ARG;
  if (dtype != CAR_BF16 && dtype != CAR_FP16 && dtype != CAR_FP32) return CAR_ERR_ARG;
  const int es = dtype == CAR_FP32 ? 4 : 2;
  if (N > (int64_t)INT32_MAX / es || (N * es) % 16 != 0) return CAR_ERR_SIZE;
  // whole message and both wire formats must stay far below int64 range
  if (M > ((int64_t)1 << 56) / (N * es)) return CAR_ERR_SIZE;
  const int64_t D = M * N * es;
  if ((D + 119) / 120 > (int64_t)UINT32_MAX || D / 8 > (int64_t)UINT32_MAX) return CAR_ERR_SIZE;

  car_ctx* h = new (std::nothrow) car_ctx();
  if (!h) return CAR_ERR_ARG;
  h->W = W;
  h->M = M;
  h->N = N;
  h->dtype = (int)dtype;
  h->es = es;
  h->D = D;
  h->nvec = D / 16;
  h->vec_per_row = (int)(N * es / 16);
  h->ll128_lines = (D + 119) / 120;
  h->ll_lines = D / 8;
  h->hook = car::WaitHook{car::kWaitLimitNs, 0, 0, -1};

  auto fail = [&](cudaError_t e, const char* where) {
    for (auto*& p : h->log)
      if (p) cudaFree(p);
    if (h->d_err) cudaFree(h->d_err);
    delete h;
    return cuda_fail(e, where);
  };
  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) return fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) return fail(e, "SM count");

  int per_sm = 0, per_sm2 = 0;
  if ((e = car::reduce_occupancy(h->dtype, W, &per_sm)) != cudaSuccess) return fail(e, "reduce occupancy");
  const int64_t per_cta = (int64_t)car::kReduceThreads * car::reduce_vectors_per_thread(W);
  h->reduce_grid = clamp_grid((h->nvec + per_cta - 1) / per_cta, per_sm, h->num_sms);
  if ((e = car::two_shot_occupancy(h->dtype, W, &per_sm)) != cudaSuccess) return fail(e, "two-shot occupancy");
  h->two_shot_grid = clamp_grid((h->nvec + per_cta - 1) / per_cta, per_sm, h->num_sms);

  const int64_t pairs = (h->ll128_lines + 1) / 2;
  const int64_t warps_needed = (pairs + 1) / 2;
  const int64_t blocks_needed = (warps_needed + car::kWireThreads / 32 - 1) / (car::kWireThreads / 32);
  for (int mis = 0; mis < 2; mis++) {
    if ((e = car::ll128_occupancy(h->dtype, W, mis != 0, h->ll128_lines, &per_sm, &per_sm2)) != cudaSuccess)
      return fail(e, "ll128 occupancy");
    h->ll128_decode_grid[mis] = clamp_grid(blocks_needed, per_sm, h->num_sms);
    h->ll128_encode_grid[mis] = clamp_grid(blocks_needed, per_sm2, h->num_sms);
  }

  if ((e = car::ll_occupancy(h->dtype, W, &per_sm, &per_sm2)) != cudaSuccess) return fail(e, "ll occupancy");
  h->ll_decode_grid = clamp_grid((h->ll_lines + car::kWireThreads - 1) / car::kWireThreads, per_sm, h->num_sms);
  h->ll_encode_grid = clamp_grid((h->nvec + car::kWireThreads - 1) / car::kWireThreads, per_sm2, h->num_sms);

  h->fused_ok = N * es <= (int64_t)CAR_MAX_ROW_BYTES;
  // The pipelined kernel takes whole rows by default: splitting rows over CTA
  // pairs puts a cross-SM exchange on every row's critical path, which
  // measured slower on GB300 than the quantisation it removes.
  h->tma_ok = h->fused_ok && car::fused_tma_shape(M, h->vec_per_row, h->num_sms, 1, W, &h->tma);
  h->tma_auto = h->tma;
  if (h->tma_ok && (e = car::fused_tma_prepare(h->dtype, W, h->tma)) != cudaSuccess) return fail(e, "pipeline smem");
  h->fused_kernel_auto = auto_fused_kernel(h);
  h->fused_kernel = h->fused_kernel_auto;
  if (h->fused_ok) {
    h->fused_auto = auto_fused_shape(W, M, h->vec_per_row, h->num_sms);
    car_status st = finish_fused_shape(h, h->fused_auto);
    if (st != CAR_OK) {
      delete h;
      return st;
    }
    h->fused_auto = h->fused;
  }

  h->lamport_ok = h->fused_ok && dtype == CAR_BF16;
  if (h->lamport_ok) {
    car::FusedShape sh = auto_lamport_shape(W, M, h->vec_per_row, h->num_sms);
    int groups = 0;
    if ((e = car::lamport_resident_groups(W, sh, h->num_sms, &groups)) != cudaSuccess) return fail(e, "lamport occupancy");
    sh.groups = (int)std::max<int64_t>(1, std::min<int64_t>(M, std::max(groups, 1)));
    h->lamport = sh;
    h->lamport_grid = clamp_grid((h->nvec + car::kWireThreads - 1) / car::kWireThreads, 8, h->num_sms);
  }
  e = cudaMalloc(reinterpret_cast<void**>(&h->d_err), 16);
  if (e != cudaSuccess) return fail(e, "cudaMalloc error word");
  e = cudaMemset(h->d_err, 0, 16);
  if (e != cudaSuccess) return fail(e, "cudaMemset error word");
  for (int k = 0; k < 3; k++) {
    e = cudaMalloc(reinterpret_cast<void**>(&h->log[k]), sizeof(car::StaleLog));
    if (e != cudaSuccess) return fail(e, "cudaMalloc stale log");
    e = cudaMemset(h->log[k], 0, sizeof(unsigned long long) * 2);
    if (e != cudaSuccess) return fail(e, "cudaMemset stale log");
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_live.insert(h);
  }
  *out = h;
  return CAR_OK;
}

car_status car_destroy(car_ctx* h) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!h || g_live.erase(h) == 0) return CAR_ERR_HANDLE;
  }
  car_status st = CAR_OK;
  for (auto* p : h->log) {
    cudaError_t e = cudaFree(p);
    if (e != cudaSuccess && st == CAR_OK) st = cuda_fail(e, "cudaFree");
  }
  cudaError_t e = cudaFree(h->d_err);
  if (e != cudaSuccess && st == CAR_OK) st = cuda_fail(e, "cudaFree");
  delete h;
  return st;
}

car_status car_tune_fused(car_ctx* h, int kernel, int cluster, int threads, int vpt) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  if (!h->fused_ok) return CAR_ERR_SIZE;
  if (kernel == CAR_FUSED_AUTO) {
    if (cluster || threads || vpt) return CAR_ERR_ARG;
    h->fused_kernel = h->fused_kernel_auto;
    h->tma = h->tma_auto;
    return finish_fused_shape(h, h->fused_auto);
  }
  if (kernel == CAR_FUSED_PIPELINE) {
    if (threads || vpt || (cluster != 0 && cluster != 1 && cluster != 2)) return CAR_ERR_ARG;
    if (!h->tma_ok) return CAR_ERR_SIZE;
    car::FusedTmaShape t;
    if (!car::fused_tma_shape(h->M, h->vec_per_row, h->num_sms, cluster ? cluster : 1, h->W, &t)) return CAR_ERR_SIZE;
    cudaError_t e = car::fused_tma_prepare(h->dtype, h->W, t);
    if (e != cudaSuccess) return cuda_fail(e, "pipeline smem");
    h->tma = t;
    h->fused_kernel = CAR_FUSED_PIPELINE;
    return CAR_OK;
  }
  if (kernel != CAR_FUSED_ROWS) return CAR_ERR_ARG;
  car::FusedShape sh = h->fused_auto;
  if (cluster) sh.cluster = cluster;
  if (threads) sh.threads = threads;
  if (vpt) sh.vpt = vpt;
  if (sh.cluster != 1 && sh.cluster != 2 && sh.cluster != 4 && sh.cluster != 8) return CAR_ERR_ARG;
  if (!car::fused_has_variant(h->W, sh.vpt)) return CAR_ERR_ARG;
  if (sh.threads < 32 || sh.threads % 32 || sh.threads > car::fused_max_threads(h->W, sh.vpt)) return CAR_ERR_ARG;
  if (!shape_valid(h->W, h->vec_per_row, sh)) return CAR_ERR_SIZE;
  st = finish_fused_shape(h, sh);
  if (st == CAR_OK) h->fused_kernel = CAR_FUSED_ROWS;
  return st;
}

car_status car_test_delay_partial(car_ctx* h, uint64_t wait_limit_ns, int cta, int64_t row, uint64_t delay_ns) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  if (cta < 0) {
    if (wait_limit_ns || row || delay_ns) return CAR_ERR_ARG;
    h->hook = car::WaitHook{car::kWaitLimitNs, 0, 0, -1};
    return CAR_OK;
  }
  if (cta > 7 || row < 0 || row >= h->M || wait_limit_ns < 1000 || wait_limit_ns > car::kWaitLimitNs ||
      delay_ns > CAR_TEST_MAX_DELAY_NS)
    return CAR_ERR_ARG;
  h->hook = car::WaitHook{wait_limit_ns, delay_ns, row, cta};
  return CAR_OK;
}

car_status car_sync(car_ctx* h, void* stream) {
  if (!live(h)) return CAR_ERR_HANDLE;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int err = 0;
  e = cudaMemcpy(&err, h->d_err, sizeof(err), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (!err) return CAR_OK;
  e = cudaMemset(h->d_err, 0, sizeof(err));
  if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  snprintf(g_err, sizeof(g_err), "a kernel gave up a bounded wait (code %u)", err);
  return CAR_ERR_TIMEOUT;
}

car_status car_reduce(car_ctx* h, const void* const* inputs, void* ar_out, void* stream) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  car::RankPtrs tbl;
  if ((st = check_table(h, inputs, &tbl)) != CAR_OK) return st;
  if ((st = check_dev(ar_out)) != CAR_OK) return st;
  cudaError_t e = car::launch_reduce(h->dtype, h->W, tbl, ar_out, h->nvec, h->reduce_grid,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "rank_sum_reduce launch");
}

car_status car_reduce_two_shot(car_ctx* h, const void* const* inputs, void* ar_out, void* stream) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  car::RankPtrs tbl;
  if ((st = check_table(h, inputs, &tbl)) != CAR_OK) return st;
  if ((st = check_dev(ar_out)) != CAR_OK) return st;
  cudaError_t e = car::launch_two_shot(h->dtype, h->W, tbl, ar_out, h->nvec, h->two_shot_grid,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "rank_sum_two_shot launch");
}

car_status car_reduce_residual_rmsnorm(car_ctx* h, const void* const* inputs, const void* residual,
                                       const void* weight, float eps, void* residual_out,
                                       void* norm_out, void* ar_out, void* stream) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  if (!std::isfinite(eps) || eps < 0.f) return CAR_ERR_ARG;
  car::RankPtrs tbl;
  if ((st = check_table(h, inputs, &tbl)) != CAR_OK) return st;
  if ((st = check_dev(residual)) != CAR_OK) return st;
  if ((st = check_dev(weight)) != CAR_OK) return st;
  if ((st = check_dev(residual_out)) != CAR_OK) return st;
  if ((st = check_dev(norm_out)) != CAR_OK) return st;
  if (ar_out && !aligned16(ar_out)) return CAR_ERR_ALIGN;
  if (!h->fused_ok) return CAR_ERR_SIZE;
  cudaError_t e;
  if (h->fused_kernel == CAR_FUSED_PIPELINE)
    e = car::launch_fused_tma(h->dtype, h->W, tbl, residual, weight, eps, residual_out, norm_out, ar_out,
                              h->d_err, h->M, h->N, h->vec_per_row, h->tma, static_cast<cudaStream_t>(stream));
  else
    e = car::launch_fused(h->dtype, h->W, tbl, residual, weight, eps, residual_out, norm_out, ar_out, h->d_err,
                          h->M, h->N, h->vec_per_row, h->fused, h->hook, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "reduce_residual_rmsnorm launch");
}

size_t car_ll128_wire_bytes(car_ctx* h) { return live(h) ? (size_t)(128 * h->ll128_lines) : 0; }
size_t car_ll_wire_bytes(car_ctx* h) { return live(h) ? (size_t)(16 * h->ll_lines) : 0; }

car_status car_ll128_encode(car_ctx* h, const void* data, uint64_t flag, void* wire, void* stream) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  if ((st = check_dev_elem(data, h->es)) != CAR_OK) return st;
  if ((st = check_dev(wire)) != CAR_OK) return st;
  const int mis = aligned16(data) ? 0 : 1;
  cudaError_t e = car::launch_ll128_encode(data, h->D, h->ll128_lines, flag, wire, h->ll128_encode_grid[mis],
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "ll128_encode launch");
}

car_status car_ll128_decode_reduce(car_ctx* h, const void* const* wires, uint64_t expected_flag,
                                   int max_polls, void* ar_out, void* stream) {
  car::RankPtrs tbl;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  car_status st = decode_common(h, 0, wires, max_polls, ar_out, s, &tbl);
  if (st != CAR_OK) return st;
  cudaError_t e = car::launch_ll128_decode_reduce(h->dtype, h->W, tbl, h->D, h->ll128_lines, expected_flag,
                                                  max_polls, ar_out, h->log[0], next_log_slot(h, 0),
                                                  h->ll128_decode_grid[aligned16(ar_out) ? 0 : 1], s);
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "ll128_decode_reduce launch");
}

car_status car_ll128_report(car_ctx* h, car_stale_report* out) { return report_common(h, 0, out); }

car_status car_ll_encode(car_ctx* h, const void* data, uint32_t flag, void* wire, void* stream) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  if ((st = check_dev(data)) != CAR_OK) return st;
  if ((st = check_dev(wire)) != CAR_OK) return st;
  cudaError_t e = car::launch_ll_encode(data, h->D, flag, wire, h->ll_encode_grid,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "ll_encode launch");
}

car_status car_ll_decode_reduce(car_ctx* h, const void* const* wires, uint32_t expected_flag,
                                int max_polls, void* ar_out, void* stream) {
  car::RankPtrs tbl;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  car_status st = decode_common(h, 1, wires, max_polls, ar_out, s, &tbl);
  if (st != CAR_OK) return st;
  cudaError_t e = car::launch_ll_decode_reduce(h->dtype, h->W, tbl, h->D, expected_flag, max_polls,
                                               ar_out, h->log[1], next_log_slot(h, 1), h->ll_decode_grid, s);
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "ll_decode_reduce launch");
}

car_status car_ll_report(car_ctx* h, car_stale_report* out) { return report_common(h, 1, out); }

size_t car_lamport_buffer_bytes(car_ctx* h) {
  return (live(h) && h->dtype == CAR_BF16) ? (size_t)(3 * (int64_t)h->W * h->D) : 0;
}

static car_status lamport_checks(car_ctx* h, const void* comm) {
  car_status st = check_handle(h);
  if (st != CAR_OK) return st;
  if (h->dtype != CAR_BF16) {
    snprintf(g_err, sizeof(g_err), "the Lamport format packs bf16 pairs: the handle's dtype must be bf16");
    return CAR_ERR_ARG;
  }
  if (!h->lamport_ok) return CAR_ERR_SIZE;
  return check_dev(comm);
}

car_status car_lamport_init(car_ctx* h, void* comm, void* stream) {
  car_status st = lamport_checks(h, comm);
  if (st != CAR_OK) return st;
  cudaError_t e = car::launch_lamport_fill(comm, 3 * (int64_t)h->W * h->D, h->lamport_grid,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "lamport fill launch");
}

car_status car_lamport_push(car_ctx* h, const void* data, int rank, uint64_t round, void* comm, void* stream) {
  car_status st = lamport_checks(h, comm);
  if (st != CAR_OK) return st;
  if (rank < 0 || rank >= h->W) return CAR_ERR_ARG;
  if ((st = check_dev(data)) != CAR_OK) return st;
  uint8_t* slot = static_cast<uint8_t*>(comm) + ((int64_t)(round % 3) * h->W + rank) * h->D;
  cudaError_t e = car::launch_lamport_push(data, h->D, slot, h->lamport_grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "lamport push launch");
}

car_status car_lamport_reduce_residual_rmsnorm(car_ctx* h, void* comm, uint64_t round, int max_polls,
                                               const void* residual, const void* weight, float eps,
                                               void* residual_out, void* norm_out, void* ar_out, void* stream) {
  car_status st = lamport_checks(h, comm);
  if (st != CAR_OK) return st;
  if (max_polls < 1 || !std::isfinite(eps) || eps < 0.f) return CAR_ERR_ARG;
  if ((st = check_dev(residual)) != CAR_OK) return st;
  if ((st = check_dev(weight)) != CAR_OK) return st;
  if ((st = check_dev(residual_out)) != CAR_OK) return st;
  if ((st = check_dev(norm_out)) != CAR_OK) return st;
  if (ar_out && !aligned16(ar_out)) return CAR_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->last_stream[2] = s;
  h->decoded[2] = true;
  cudaError_t e;
  const int64_t region_bytes = (int64_t)h->W * h->D;
  uint8_t* base = static_cast<uint8_t*>(comm);
  e = car::launch_lamport_reduce(h->W, base + (int64_t)(round % 3) * region_bytes,
                                 base + (int64_t)((round + 2) % 3) * region_bytes, h->D, residual, weight, eps,
                                 residual_out, norm_out, ar_out, h->log[2], next_log_slot(h, 2), max_polls,
                                 h->d_err, h->M, h->N, h->vec_per_row, h->lamport, s);
  return e == cudaSuccess ? CAR_OK : cuda_fail(e, "lamport receive launch");
}

car_status car_lamport_report(car_ctx* h, car_stale_report* out) { return report_common(h, 2, out); }

}  // extern "C"
