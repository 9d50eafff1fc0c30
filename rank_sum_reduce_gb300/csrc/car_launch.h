// car_launch.h -- host-side launch entry points of libcar's kernels (internal).
// Argument checking lives in api.cu; these functions only pick the template
// instance for (dtype, W) and launch it on the given stream.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace car {

struct RankPtrs;
struct StaleLog;

// ---- plain one-shot rank sum (reduce.cu) ----
// nvec = number of 16-byte vectors per rank.  grid = CTAs of kReduceThreads.
constexpr int kReduceThreads = 256;
int reduce_vectors_per_thread(int W);
cudaError_t reduce_occupancy(int dtype, int W, int* blocks_per_sm);
cudaError_t launch_reduce(int dtype, int W, const RankPtrs& in, void* out, int64_t nvec, int grid,
                          cudaStream_t s);
// two-shot bit pattern: shard s of the nvec units summed from rank s onwards
cudaError_t two_shot_occupancy(int dtype, int W, int* blocks_per_sm);
cudaError_t launch_two_shot(int dtype, int W, const RankPtrs& in, void* out, int64_t nvec, int grid,
                            cudaStream_t s);

// ---- fused rank sum + residual + RMSNorm (fused.cu) ----
struct FusedShape {
  int cluster;  // CTAs per row (1, 2, 4, 8)
  int threads;  // threads per CTA
  int vpt;      // 16-byte vectors per thread (1, 2, 4)
  int groups;   // row groups in the grid (grid = groups * cluster)
};
// Largest CTA the (W, vpt) instance is compiled for, and whether it exists
// (vpt 2 exists for W in {1, 2, 4, 8}; vpt 1 for every W).
int fused_max_threads(int W, int vpt);
bool fused_has_variant(int W, int vpt);
// How many row groups of this shape can be resident at once (0 on error).
cudaError_t fused_resident_groups(int dtype, int W, const FusedShape& sh, int num_sms, int* groups);
// The split-row partial exchange's wait limit, and the test hook that makes
// one CTA push its partial late (delay_cta < 0: none).
struct WaitHook {
  unsigned long long wait_ns;
  unsigned long long delay_ns;
  int64_t delay_row;
  int delay_cta;
};
cudaError_t launch_fused(int dtype, int W, const RankPtrs& in, const void* residual,
                         const void* weight, float eps, void* residual_out, void* norm_out,
                         void* ar_out, unsigned int* err, int64_t rows, int64_t cols, int vec_per_row,
                         const FusedShape& sh, const WaitHook& hook, cudaStream_t s);

// ---- fused, many rows: TMA bulk copies into a shared-memory ring (fused_tma.cu) ----
struct FusedTmaShape {
  int cluster;    // CTAs sharing each row (1 or 2)
  int ls;         // trailing slices of a row loaded by the consumers, not bulk-copied (0 or 3)
  int consumers;  // consumer threads (the CTA adds one producer warp)
  int vpt;        // 16-byte vectors per consumer thread (1, 2, 4, 8)
  int slots;      // ring depth in row slices
  int grid;       // persistent CTAs
  int smem;       // dynamic shared memory bytes
};
// False when the row does not fit the ring design.
bool fused_tma_shape(int64_t rows, int vec_per_row, int num_sms, int cluster, int W, FusedTmaShape* out);
// Once per shape: allow the kernel instance its dynamic shared memory.
cudaError_t fused_tma_prepare(int dtype, int W, const FusedTmaShape& sh);
cudaError_t launch_fused_tma(int dtype, int W, const RankPtrs& in, const void* residual, const void* weight,
                             float eps, void* residual_out, void* norm_out, void* ar_out, unsigned int* err,
                             int64_t rows, int64_t cols, int vec_per_row, const FusedTmaShape& sh,
                             cudaStream_t s);

// ---- LL128 (ll128.cu) ----
constexpr int kWireThreads = 256;
// Resident CTAs per SM of the decode and encode instances that a call with
// 16-byte aligned (mis = false) or misaligned (mis = true) output / rank data
// launches on a message of `lines` LL128 lines.
// publish: the decode instance of the allocation-free entry (see ll128.cu).
cudaError_t ll128_occupancy(int dtype, int W, bool mis, int64_t lines, int* decode_blocks_per_sm,
                            int* encode_blocks_per_sm, bool publish = false);
cudaError_t launch_ll128_encode(const void* data, int64_t data_bytes, int64_t lines, uint64_t flag,
                                void* wire, int grid, cudaStream_t s);
// With a report buffer, the allocation-free instance: `log` is the shared
// array (slot unused), and the last CTA writes the count and the first `cap`
// pairs to `report` and clears the array.
cudaError_t launch_ll128_decode_reduce(int dtype, int W, const RankPtrs& wires, int64_t data_bytes,
                                       int64_t lines, uint64_t expected, int max_polls, void* out,
                                       StaleLog* log, int log_slot, int grid, cudaStream_t s,
                                       void* report = nullptr, uint32_t cap = 0);

// ---- Lamport one-shot push, bf16 (lamport.cu) ----
bool lamport_has_variant(int W, int vpt);
int lamport_max_threads(int W, int vpt);
cudaError_t lamport_resident_groups(int W, const FusedShape& sh, int num_sms, int* groups);
cudaError_t launch_lamport_fill(void* words, int64_t bytes, int grid, cudaStream_t s);
cudaError_t launch_lamport_push(const void* data, int64_t bytes, void* slot, int grid, cudaStream_t s);
cudaError_t launch_lamport_reduce(int W, const void* region, void* clear_region, int64_t slot_bytes,
                                  const void* residual, const void* weight, float eps, void* residual_out,
                                  void* norm_out, void* ar_out, StaleLog* log, int log_slot, int max_polls,
                                  unsigned int* err, int64_t rows, int64_t cols, int vec_per_row,
                                  const FusedShape& sh, cudaStream_t s);

// ---- diagnostics (api.cu): text returned by car_last_error() on this thread ----
void set_last_error(const char* msg);

// ---- LL (ll.cu) ----
cudaError_t ll_occupancy(int dtype, int W, int* decode_blocks_per_sm, int* encode_blocks_per_sm);
cudaError_t launch_ll_encode(const void* data, int64_t data_bytes, uint32_t flag, void* wire,
                             int grid, cudaStream_t s);
cudaError_t launch_ll_decode_reduce(int dtype, int W, const RankPtrs& wires, int64_t data_bytes,
                                    uint32_t expected, int max_polls, void* out, StaleLog* log, int log_slot,
                                    int grid, cudaStream_t s);

}  // namespace car
