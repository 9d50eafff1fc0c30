/*
 * oracle.h -- plain, slow, single-threaded CPU oracle for the rank-sum reduce
 * hot path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * bench's CPU-baseline leg load it; the product library never does, and it
 * shares no code, header or table with the CUDA path.
 *
 * Pages cited (title, then section):
 *   P1  "SGLang Custom AllReduce v1 线程模型和工作原理细节"
 *   P2  "NCCL 专家课程 14：Simple、LL、LL128 的线格式、同步与真实性能边界"
 *   P3  "0-custom-all-reduce" (SGLang JIT custom all-reduce notes)
 *   P4  "用 Triton + Symmetric Memory 写一个 AllReduce + RMSNorm 融合算子"
 *
 * Element types: 0 = bf16, 1 = fp16, 2 = fp32, stored little-endian.
 * Every function takes host pointers and never allocates more than O(W).
 */
#ifndef RSR_ORACLE_H
#define RSR_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_FP32 = 2 };

/* ---- scalar conversions (IEEE 754 binary formats, round half to even) ---- */
float    orc_bf16_to_f32(uint16_t b);
float    orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float f);
uint16_t orc_f32_to_f16(float f);
uint16_t orc_f64_to_bf16(double d);
uint16_t orc_f64_to_f16(double d);
float    orc_f64_to_f32(double d);
int      orc_elem_size(int dtype);
/* Array form of the conversions above, for the pins: kinds are the element
 * types plus 3 = fp64.  Widening (bf16/fp16 -> fp32/fp64, fp32 -> fp64) is
 * exact; narrowing rounds half to even.  Same-kind copies are bit copies. */
void     orc_convert(const void* src, int src_kind, void* dst, int dst_kind, int64_t n);

/* ---- one-shot rank sum: P1 "1stage：kernel 全文与时间线" (packed_reduce),
 *      P3 "4. 求和(reduce_impl)".  ar[i] = rne_T(((x_0 + x_1) + ...) + x_{W-1})
 *      with every "+" an fp32 add, seeded with x_0. n = element count. ---- */
void orc_reduce(int W, const void* const* x, int dtype, int64_t n, void* ar);

/* ---- two-shot bit pattern: P1 "2stage：分片、轮转、以及为什么没有出口 barrier".
 *      The message's 16-byte packed units are cut into W shards of
 *      part = units / W units; the last shard also takes the remainder (all
 *      units when part == 0).  Shard s is summed by its owner in the rotated
 *      order s, s+1, ..., s-1 (mod W), fp32, one rounding.  n * elem_size must
 *      be a multiple of 16 (otherwise nothing is written). ---- */
void orc_reduce_two_shot(int W, const void* const* x, int dtype, int64_t n, void* ar);

/* ---- fused reduce + residual + RMSNorm: P4 "这个算子在算什么".
 *      Row-major [M,N].  ar (nullable), residual_out, norm_out have type
 *      dtype; norm_f64 (nullable, M*N doubles) receives the unrounded value.
 *      Statistics are taken in double (the oracle's exact-as-practical
 *      reading); ar and residual_out are bit-exact fp32 definitions. ---- */
void orc_reduce_residual_rmsnorm(int W, const void* const* x, const void* residual,
                                 const void* weight, float eps, int64_t M, int64_t N,
                                 int dtype, void* ar, void* residual_out, void* norm_out,
                                 double* norm_f64);

/* ---- LL128 line format: P2 "LL128 的 128-byte line",
 *      "LL128 的 warp-level ready 检查".  A 128-byte line carries 15 data
 *      words (uint64) and one flag word (the 16th). ---- */
int64_t orc_ll128_lines(int64_t data_bytes);          /* ceil(D/120)        */
int64_t orc_ll128_wire_bytes(int64_t data_bytes);     /* 128*ceil(D/120)    */
int64_t orc_ll128_data_capacity(int64_t wire_bytes);  /* 120*(wire/128)     */
void    orc_ll128_encode(const void* data, int64_t data_bytes, uint64_t flag, void* wire);
/* Validates every (rank, line), decodes, and reduces in rank order.
 * Elements covered by a line that is stale in any rank are written as 0.
 * Stale (rank, line) pairs go to stale[k][0..1] in line-major, rank-minor
 * order, up to cap entries; the return value is the total stale count. */
int64_t orc_ll128_decode_reduce(int W, const void* const* wires, int64_t data_bytes,
                                int dtype, uint64_t expected_flag, void* ar,
                                uint32_t* stale, int64_t cap);

/* ---- LL line format: P2 "LL 的 16-byte FIFO line", "LL 如何发布和等待
 *      flag".  A 16-byte line is {data1, flag1, data2, flag2} (uint32 each)
 *      carrying one 8-byte data word. ---- */
int64_t orc_ll_lines(int64_t data_bytes);             /* ceil(D/8)          */
int64_t orc_ll_wire_bytes(int64_t data_bytes);        /* 16*ceil(D/8)       */
int64_t orc_ll_data_capacity(int64_t wire_bytes);     /* 8*(wire/16)        */
void    orc_ll_encode(const void* data, int64_t data_bytes, uint32_t flag, void* wire);
int64_t orc_ll_decode_reduce(int W, const void* const* wires, int64_t data_bytes,
                             int dtype, uint32_t expected_flag, void* ar,
                             uint32_t* stale, int64_t cap);

/* ---- Lamport one-shot push (bf16 only): P4 "方案二：Lamport（负零轮询）".
 *      A receive buffer holds 3 regions x W slots x n bf16 values and starts
 *      filled with the sentinel word 0x80008000 (two bf16 -0.0).  A push
 *      writes a rank's values into its slot of region (round % 3) with every
 *      -0.0 (0x8000) turned into +0.0, so pushed words never equal the
 *      sentinel.  The receive step treats a sentinel word as "not arrived":
 *      rows of [M, N] with a missing word in any rank are stale (outputs 0,
 *      (rank, row) pairs listed, row-major then rank order); other rows get
 *      the fused rank sum + residual + RMSNorm.  It then refills region
 *      (round + 2) % 3 -- the previous round's -- with the sentinel. ---- */
#define ORC_LAMPORT_SENTINEL 0x80008000u
void    orc_lamport_fill(void* words, int64_t n_words);
void    orc_lamport_push(const void* data, int64_t n, void* slot);
int64_t orc_lamport_reduce_residual_rmsnorm(int W, void* buffer, uint64_t round, int64_t M, int64_t N,
                                            const void* residual, const void* weight, float eps,
                                            void* ar, void* residual_out, void* norm_out,
                                            uint32_t* stale, int64_t cap);

#ifdef __cplusplus
}
#endif
#endif
