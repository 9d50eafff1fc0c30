/*
 * car.h -- C ABI of libcar: one-shot rank-sum reduce, fused residual add +
 * RMSNorm, and LL / LL128 line encode, validate and decode-reduce, for one
 * GB300 (sm_103a).
 *
 * The W "ranks" are W separate device buffers on the same GPU: they stand in
 * for the peer-mapped buffers a multi-GPU one-shot all-reduce reads.  There is
 * no cross-GPU barrier, no IPC and no transport; every entry point runs
 * hand-written CUDA kernels on the caller's stream.
 *
 * Pages the operations come from (title, then section):
 *   P1  "SGLang Custom AllReduce v1 线程模型和工作原理细节"
 *   P2  "NCCL 专家课程 14：Simple、LL、LL128 的线格式、同步与真实性能边界"
 *   P3  "0-custom-all-reduce" (SGLang JIT custom all-reduce notes)
 *   P4  "用 Triton + Symmetric Memory 写一个 AllReduce + RMSNorm 融合算子"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Shapes.  A handle fixes W (number of rank buffers, 1..16), M rows, N
 *   columns and the element type.  Every [M, N] tensor is row-major and
 *   contiguous; D = M*N*s bytes per rank (s = 2 for bf16/fp16, 4 for fp32).
 *   N*s must be a multiple of 16 so that each row starts on a 16-byte
 *   boundary (P1 "线程模型：16 字节一个单位": the message is processed in
 *   16-byte packed units; P3 "2. 线程怎么分活").
 * - Pointers.  "dev" pointers are device memory on the handle's device,
 *   owned by the caller, and must be 16-byte aligned unless the call states
 *   otherwise (the LL128 data and outputs need only element alignment).
 *   Pointer tables
 *   (inputs, wires) are host arrays of W device pointers, read during the
 *   call only.  The library never frees caller memory.
 * - Streams.  `stream` is a cudaStream_t passed as void*; NULL is the legacy
 *   default stream.  Launches are asynchronous: a CAR_OK return means the work
 *   was queued; results are valid once the stream has reached that point.
 * - Errors.  Arguments are checked before anything is queued; a failed check
 *   returns its code and launches nothing.  No entry point throws, traps,
 *   spins without bound or calls exit.  CUDA errors seen at launch return
 *   CAR_ERR_CUDA; car_last_error() gives the text.
 * - Threads.  Distinct handles may be used from distinct threads.  One
 *   handle must not be used by two threads at once.
 */
#ifndef CAR_H
#define CAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { CAR_BF16 = 0, CAR_FP16 = 1, CAR_FP32 = 2 } car_dtype;

typedef enum {
  CAR_OK = 0,
  CAR_ERR_ARG = 1,        /* NULL pointer, W/M/N/dtype out of range, bad max_polls */
  CAR_ERR_ALIGN = 2,      /* a device pointer below the alignment its call needs    */
  CAR_ERR_SIZE = 3,       /* N*s not a multiple of 16, size overflow, row too long  */
  CAR_ERR_CUDA = 4,       /* CUDA runtime error (see car_last_error)                */
  CAR_ERR_STALE_FLAG = 5, /* a decode found lines whose flag was not the expected one */
  CAR_ERR_HANDLE = 6,     /* NULL, destroyed or foreign handle                      */
  CAR_ERR_TIMEOUT = 7     /* a kernel gave up a bounded wait (see car_sync)         */
} car_status;

/* Kernels of car_reduce_residual_rmsnorm (see car_tune_fused). */
typedef enum { CAR_FUSED_AUTO = 0, CAR_FUSED_ROWS = 1, CAR_FUSED_PIPELINE = 2 } car_fused_kernel;

typedef struct car_ctx car_ctx; /* opaque */

/* Stale-line report of the last decode-reduce on a handle.  The caller sets
 * `cap` and `entries` (a host array of cap (rank, line) pairs, may be NULL
 * when cap == 0); the library fills n_stale (every stale (rank, line) pair
 * found) and n_listed (pairs written, at most min(cap, CAR_STALE_LIST_MAX)).
 * Order of the entries is unspecified; compare them as a set. */
typedef struct {
  uint64_t n_stale;
  uint32_t n_listed;
  uint32_t cap;
  uint32_t (*entries)[2];
} car_stale_report;

/* Device-side capacity of the stale list kept per handle and per format. */
#define CAR_STALE_LIST_MAX 65536u

/* Longest row the fused kernel takes: N*s <= CAR_MAX_ROW_BYTES (64 KiB,
 * e.g. N = 32768 bf16 or 16384 fp32). */
#define CAR_MAX_ROW_BYTES (64u * 1024u)

/* ---------------------------------------------------------------------- */
/* Handles                                                                 */
/* ---------------------------------------------------------------------- */

/* Create a handle for W rank buffers of [M, N] elements of `dtype` on the
 * current CUDA device.  The handle owns only its own small device scratch
 * (stale-line counters and lists, about 1 MB) and the launch shapes it picks
 * for this problem.  Errors: CAR_ERR_ARG (out == NULL, W not in 1..16, M < 1,
 * N < 1, unknown dtype), CAR_ERR_SIZE (N*s % 16 != 0, or M*N*s overflows
 * int64), CAR_ERR_CUDA (no device, allocation failed).  *out is set to NULL
 * on error. */
car_status car_create(int W, int64_t M, int64_t N, car_dtype dtype, car_ctx** out);

/* Free the handle and its scratch.  Waits for nothing: the caller must make
 * sure no queued work still uses it.  CAR_ERR_HANDLE for an unknown handle. */
car_status car_destroy(car_ctx* h);

/* ---------------------------------------------------------------------- */
/* One-shot rank sum (P1 "1stage：kernel 全文与时间线", packed_reduce;     */
/* P3 "3. 从所有 GPU 读" and "4. 求和(reduce_impl)")                       */
/* ---------------------------------------------------------------------- */

/* ar_out[i] = rne_T( (((f32(x_0[i]) + f32(x_1[i])) + ...) + f32(x_{W-1}[i])) )
 * for every element i of the [M, N] problem: fp32 adds in rank order 0..W-1,
 * seeded with rank 0's value, one round-to-nearest-even at the end (identity
 * for fp32).  The order is fixed so that every caller gets the same bits.
 *   inputs : host array of W dev pointers, each D bytes.
 *   ar_out : dev, D bytes; may equal inputs[k] for one k (each element is read
 *            before it is written, by the same thread).  Other overlap is
 *            undefined.
 * Errors: CAR_ERR_HANDLE, CAR_ERR_ARG (NULL), CAR_ERR_ALIGN, CAR_ERR_CUDA. */
car_status car_reduce(car_ctx* h, const void* const* inputs, void* ar_out, void* stream);

/* Two-shot bit pattern (P1 "2stage：分片、轮转、以及为什么没有出口 barrier"):
 * the same sum as car_reduce, but rounded as a reduce-scatter + all-gather
 * would round it.  The message's 16-byte units are cut into W shards of
 * part = units / W (the last shard also takes the remainder; all units when
 * part == 0), and shard s is summed by its owner in the rotated rank order
 * s, s+1, ..., s-1.  Arguments, aliasing and errors as car_reduce. */
car_status car_reduce_two_shot(car_ctx* h, const void* const* inputs, void* ar_out, void* stream);

/* ---------------------------------------------------------------------- */
/* Fused rank sum + residual add + RMSNorm                                 */
/* (P4 "这个算子在算什么" and "总体设计")                                   */
/* ---------------------------------------------------------------------- */

/* Per row m and column j:
 *   acc      = fp32 rank sum as in car_reduce (unrounded)
 *   h        = acc + f32(residual[m,j])               (fp32 add)
 *   residual_out[m,j] = rne_T(h);  ar_out[m,j] = rne_T(acc) when ar_out != NULL
 *   rms      = rsqrt( (sum_j h^2) / N + eps )          (fp32, any order)
 *   norm_out[m,j]     = rne_T( (h * rms) * f32(weight[j]) )
 * ar and residual_out are bit-exact; norm_out depends on the order of the
 * sum of squares and on rsqrtf, and lies within 2^-7*|ref| + 1e-5 of the
 * exactly computed value.
 *   inputs       : host array of W dev pointers, each [M, N].
 *   residual     : dev [M, N].       weight : dev [N].
 *   eps          : fp32 (e.g. 1e-6).
 *   residual_out : dev [M, N]; may equal residual.
 *   norm_out     : dev [M, N].
 *   ar_out       : dev [M, N] or NULL; may equal inputs[k].
 * Errors: CAR_ERR_HANDLE, CAR_ERR_ARG (NULL, eps not finite or < 0),
 * CAR_ERR_ALIGN, CAR_ERR_SIZE (N*s > CAR_MAX_ROW_BYTES), CAR_ERR_CUDA. */
car_status car_reduce_residual_rmsnorm(car_ctx* h, const void* const* inputs, const void* residual,
                                       const void* weight, float eps, void* residual_out,
                                       void* norm_out, void* ar_out, void* stream);

/* ---------------------------------------------------------------------- */
/* LL128 (P2 "LL128 的 128-byte line", "LL128 的 warp-level ready 检查")    */
/* ---------------------------------------------------------------------- */

/* Wire size of one rank's message: 128 * ceil(D / 120) bytes; 0 for an
 * invalid handle. */
size_t car_ll128_wire_bytes(car_ctx* h);

/* Encode one rank's D data bytes into LL128 lines: line k holds data words
 * 15k..15k+14 (uint64, little-endian, zero past the end of the data) in
 * words 0..14 and `flag` in word 15.
 *   data : dev, D bytes, aligned to the element size only: a buffer at a
 *          2..14-byte offset from a 16-byte boundary is read with aligned
 *          16-byte loads of the blocks that hold it and realigned in registers
 *          (P2 "LL128 对齐为何重要" measures NCCL's misaligned path).
 *   wire : dev, car_ll128_wire_bytes(h) bytes, 16-byte aligned.
 * Errors: CAR_ERR_HANDLE, CAR_ERR_ARG, CAR_ERR_ALIGN, CAR_ERR_CUDA. */
car_status car_ll128_encode(car_ctx* h, const void* data, uint64_t flag, void* wire, void* stream);

/* Validate, decode and reduce W LL128 wires (ar_out, like the encode's data,
 * needs only element alignment; no byte outside ar_out[0, D) is written):
 * line k of rank r is valid when
 * its word 15 equals expected_flag.  A line found stale is checked again up
 * to max_polls - 1 more times (re-reading the whole line each time); there
 * is no unbounded wait.  For every line valid in all ranks, each element of
 * its 120 data bytes is reduced as in car_reduce; the elements of a line
 * stale in any rank are written as 0, and every stale (rank, line) pair is
 * recorded for car_ll128_report.
 *   wires   : host array of W dev pointers, each car_ll128_wire_bytes(h).
 *   ar_out  : dev, D bytes.
 *   max_polls : >= 1 (1 = check once).
 * Errors: CAR_ERR_HANDLE, CAR_ERR_ARG (NULL, max_polls < 1), CAR_ERR_ALIGN,
 * CAR_ERR_CUDA.  Stale lines are reported by car_ll128_report, not here. */
car_status car_ll128_decode_reduce(car_ctx* h, const void* const* wires, uint64_t expected_flag,
                                   int max_polls, void* ar_out, void* stream);

/* Wait for the stream of the last car_ll128_decode_reduce on this handle and
 * fill *out.  Returns CAR_ERR_STALE_FLAG when n_stale > 0, CAR_OK when none
 * (or when no decode has run), CAR_ERR_HANDLE / CAR_ERR_ARG / CAR_ERR_CUDA.
 * Reading the report clears its count: a decode captured in a CUDA graph and
 * replayed reports each replay's stale lines when the report follows each
 * replay (replays without a report in between add up), and a second report
 * with no decode in between finds none.  The report waits only for the stream
 * the decode was issued (or captured) on: after a graph replay on another
 * stream, wait for that stream first. */
car_status car_ll128_report(car_ctx* h, car_stale_report* out);

/* Allocation-free variant of car_ll128_decode_reduce.  The pages have no
 * counterpart to it: it exists for callers that cannot call cudaMalloc and
 * therefore cannot create a handle (car_create allocates the handle's
 * stale-line log).  Examples: code running inside an allocator's own
 * callbacks, processes whose caching pool already holds all free device
 * memory, and latency-critical paths that cannot take the device-wide
 * synchronisation an allocation or free can cause.
 *
 * It needs no handle and allocates nothing.  Its stale-line log is a fixed
 * device array inside the library (CAR_STALE_LIST_MAX pairs, 512 KiB plus
 * two 8-byte counts) that every GPU which loads the library keeps until the
 * process exits.  The first call on a device looks up that array's device
 * address and the device's SM count, with the device current; make that
 * first call before any stream capture on the device.  The address is kept
 * for the life of the process, so the device must not be reset
 * (cudaDeviceReset) after that first call: a reset can place the array
 * elsewhere, and the kept address would then point at other memory.
 *
 * Each call is one kernel launch.  The last of its CTAs to finish copies the
 * report into stale_out and clears the array's counts for the next call, so
 * calls queued one after another on one stream (or replayed from a CUDA
 * graph) each report their own stale lines.  Every call on a device shares
 * the array: calls that overlap on the GPU (two streams at once) race on it
 * and their reports are wrong.
 *
 * Arguments: the shape (W, M, N, dtype) and data as for car_create and
 * car_ll128_decode_reduce (wires: W dev pointers of 128*ceil(M*N*s/120)
 * bytes, 16-byte aligned; ar_out: dev, M*N*s bytes, element-aligned).
 * stale_out: dev, 16-byte aligned,
 * 16 + 8*cap bytes; after the call completes on `stream` it holds the
 * uint64 count of stale (rank, line) pairs at byte 0, 8 reserved bytes, then
 * min(count, cap) pairs of uint32 (rank, line) (bytes past those are
 * leftovers).  cap may not exceed CAR_STALE_LIST_MAX.
 * Errors: CAR_ERR_ARG (shape, NULL, max_polls < 1, device index > 63),
 * CAR_ERR_SIZE (cap > CAR_STALE_LIST_MAX, with text in car_last_error(), or
 * the shape rules of car_create), CAR_ERR_ALIGN, CAR_ERR_CUDA. */
car_status car_ll128_decode_reduce_noalloc(int W, int64_t M, int64_t N, car_dtype dtype,
                                           const void* const* wires, uint64_t expected_flag,
                                           int max_polls, void* ar_out, void* stale_out,
                                           uint32_t cap, void* stream);

/* ---------------------------------------------------------------------- */
/* LL (P2 "LL 的 16-byte FIFO line", "LL 如何发布和等待 flag")              */
/* ---------------------------------------------------------------------- */

/* Wire size of one rank's message: 16 * ceil(D / 8) bytes; 0 for an invalid
 * handle. */
size_t car_ll_wire_bytes(car_ctx* h);

/* Encode: line i = {low 32 bits of data word i, flag, high 32 bits, flag}.
 *   data : dev, D bytes.   wire : dev, car_ll_wire_bytes(h) bytes. */
car_status car_ll_encode(car_ctx* h, const void* data, uint32_t flag, void* wire, void* stream);

/* Validate (both flags must equal expected_flag), decode (data1 +
 * (data2 << 32)) and reduce W LL wires; same polling, zeroing and reporting
 * rules as car_ll128_decode_reduce, with 8 data bytes per line. */
car_status car_ll_decode_reduce(car_ctx* h, const void* const* wires, uint32_t expected_flag,
                                int max_polls, void* ar_out, void* stream);

/* Report of the last car_ll_decode_reduce, as car_ll128_report. */
car_status car_ll_report(car_ctx* h, car_stale_report* out);

/* ---------------------------------------------------------------------- */
/* Lamport one-shot push, bf16 (P4 "方案二：Lamport（负零轮询）")           */
/* ---------------------------------------------------------------------- */
/* The data itself signals arrival: two bf16 share a 32-bit word, the
 * receive buffer starts filled with the sentinel word 0x80008000 (two
 * bf16 -0.0), and senders turn -0.0 into +0.0 so that real data never equals
 * it.  Buffers rotate over three regions: round k uses region k % 3 and its
 * receive step refills region (k + 2) % 3, the one round k - 1 used.
 *
 * The receive buffer `comm` (dev, car_lamport_buffer_bytes(h) bytes) holds
 * 3 regions x W slots x D bytes; slot r of region k starts at byte
 * (k * W + r) * D.  The handle's dtype must be bf16 (CAR_ERR_ARG otherwise). */

/* 3 * W * D bytes; 0 for an invalid handle or a dtype other than bf16. */
size_t car_lamport_buffer_bytes(car_ctx* h);

/* Fill all three regions with the sentinel (once, before the first round). */
car_status car_lamport_init(car_ctx* h, void* comm, void* stream);

/* Rank `rank` (0..W-1) sends its [M, N] bf16 data for round `round`: the data,
 * with -0.0 turned into +0.0, goes to slot `rank` of region round % 3. */
car_status car_lamport_push(car_ctx* h, const void* data, int rank, uint64_t round, void* comm, void* stream);

/* Receive round `round` and apply the fused op: every word of region
 * round % 3 is checked against the sentinel on the load that reads it; a
 * missing word is re-read at most max_polls - 1 more times.  Rows complete in
 * every rank get the rank sum (rank order, fp32) + residual + RMSNorm exactly
 * as car_reduce_residual_rmsnorm computes it on the pushed values; rows with
 * a word still missing in some rank are written as 0 (ar, residual_out,
 * norm_out) and every such (rank, row) is recorded for car_lamport_report.
 * Region (round + 2) % 3 is refilled with the sentinel in the same pass.
 * Arguments as car_reduce_residual_rmsnorm; max_polls >= 1. */
car_status car_lamport_reduce_residual_rmsnorm(car_ctx* h, void* comm, uint64_t round, int max_polls,
                                               const void* residual, const void* weight, float eps,
                                               void* residual_out, void* norm_out, void* ar_out, void* stream);

/* Stale (rank, row) pairs of the last Lamport receive, as car_ll128_report. */
car_status car_lamport_report(car_ctx* h, car_stale_report* out);

/* ---------------------------------------------------------------------- */
/* Diagnostics                                                              */
/* ---------------------------------------------------------------------- */

/* Static text for a status code. */
const char* car_status_string(car_status s);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* car_last_error(void);

/* Choose the kernel of car_reduce_residual_rmsnorm for this handle (tuning
 * and tests).  CAR_FUSED_ROWS: rows split over a cluster of cluster CTAs
 * (1, 2, 4 or 8) of `threads` threads (multiple of 32, at most 1024 for
 * W <= 4 with vpt 1, else 512), each thread holding vpt 16-byte vectors (1,
 * or 2 when W is 1, 2, 4 or 8); 0 for a field keeps the automatic choice.
 * CAR_FUSED_PIPELINE: one persistent CTA per SM streaming (row, rank) slices
 * into a shared-memory ring with TMA bulk copies; cluster 0 or 1 gives each
 * CTA whole rows, 2 splits every row over a CTA pair (needs an even number of
 * 16-byte columns); threads and vpt must be 0; needs N*s <= 100 KiB per CTA.
 * CAR_FUSED_AUTO (all fields 0) restores the automatic choice: the pipeline
 * with whole rows when M exceeds the SM count and a row is larger than 8 KB
 * (N*s > 8192), else rows: a row split over a
 * cluster of 8 or 4 CTAs while each CTA keeps at least 128 16-byte vectors,
 * the CTAs fit in 7/8 of the SMs, and M <= 16 or a row brings at least 48 KB
 * of inputs; one CTA per row otherwise (with two vectors per thread where
 * one vector per thread would need 1024 threads).
 * Errors: CAR_ERR_ARG for values out of range, CAR_ERR_SIZE when the shape
 * does not cover a row or the row does not fit the ring. */
car_status car_tune_fused(car_ctx* h, int kernel, int cluster, int threads, int vpt);

/* Wait for `stream` and report whether any kernel of this handle gave up one
 * of its bounded waits since the last car_sync (CAR_ERR_TIMEOUT; the flag is
 * then cleared).  Each wait is bounded to about one second: the pipelined
 * fused kernel's waits on its shared-memory barriers (it then stops and
 * leaves its remaining rows unwritten), and the waits of the fused row kernel
 * and the Lamport receive for the partials of a split row's other CTAs (each
 * thread waits for itself: the row's norm_out is then NaN in the columns of
 * every thread whose wait ran out, or those columns of the Lamport row are
 * zeroed and the row is reported stale for every rank).  None of these waits
 * runs out unless a CTA of the same launch has stopped making progress. */
car_status car_sync(car_ctx* h, void* stream);

/* Test hook for the bounded wait of the fused row kernel (CAR_FUSED_ROWS
 * with rows split over a cluster).  The pages have no such call: it serves
 * the tests of the failure path that P2 "LL 如何发布和等待 flag" gives every
 * spin (a wait that checks for abort instead of spinning forever).
 *
 * With cta in 0..7: the split row's partial exchange waits at most
 * wait_limit_ns (1000 .. 1e9) instead of about one second, and CTA `cta` of
 * the cluster that takes row `row` (0 .. M-1) reaches that row's exchange,
 * and so pushes its partial, delay_ns (at most CAR_TEST_MAX_DELAY_NS) late.
 * A thread of a peer whose wait runs out first sets the handle's error flag
 * (car_sync then returns CAR_ERR_TIMEOUT), writes NaN for its columns of that
 * row's norm_out, and then waits (bounded by about one second) until the late
 * partial has landed before it goes on, so no partial reaches a CTA that has
 * exited.  Every other output is
 * unaffected.  With cta = -1 (and the other arguments 0) the default returns.
 * Errors: CAR_ERR_ARG for values out of range, CAR_ERR_HANDLE. */
#define CAR_TEST_MAX_DELAY_NS 100000000ull /* 100 ms */
car_status car_test_delay_partial(car_ctx* h, uint64_t wait_limit_ns, int cta, int64_t row, uint64_t delay_ns);

#ifdef __cplusplus
}
#endif
#endif /* CAR_H */
