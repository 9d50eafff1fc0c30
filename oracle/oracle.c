/*
 * oracle.c -- plain, slow, single-threaded CPU oracle (TEST INFRASTRUCTURE).
 *
 * Only the tests, the smoke check and the bench's CPU-baseline leg use this
 * file.  It shares no code with the CUDA library and follows the pages'
 * definitions step by step, in their order, with no blocking or fusion:
 *
 *   P1  "SGLang Custom AllReduce v1 线程模型和工作原理细节"
 *   P2  "NCCL 专家课程 14：Simple、LL、LL128 的线格式、同步与真实性能边界"
 *   P3  "0-custom-all-reduce" (SGLang JIT custom all-reduce notes)
 *   P4  "用 Triton + Symmetric Memory 写一个 AllReduce + RMSNorm 融合算子"
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math, so
 * every float "+" is one IEEE binary32 add with round-half-to-even and
 * subnormals kept).
 *
 * Parity pins live in tests/test_oracle_pins.py: closed forms, library
 * routines for the conversions, brute force on small inputs and the values
 * the pages print.  No function here is unpinned.
 */
#include "oracle.h"

#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* little-endian byte access (explicit, so the result never depends on the  */
/* host's byte order or on the signedness of char)                          */
/* ------------------------------------------------------------------------ */
static uint16_t ld16(const uint8_t* p) { return (uint16_t)(p[0] | ((uint16_t)p[1] << 8)); }
static uint32_t ld32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
static uint64_t ld64(const uint8_t* p) { return (uint64_t)ld32(p) | ((uint64_t)ld32(p + 4) << 32); }
static void st16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void st32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}
static void st64(uint8_t* p, uint64_t v) { st32(p, (uint32_t)v); st32(p + 4, (uint32_t)(v >> 32)); }

/* ------------------------------------------------------------------------ */
/* IEEE 754 rounding, written from the definition: an exact value           */
/* (-1)^neg * sig * 2^e is rounded to the nearest number of the target      */
/* binary format, ties to the even significand; overflow gives infinity,    */
/* results below the normal range become subnormals (gradual underflow).    */
/* ------------------------------------------------------------------------ */
typedef struct {
  int p;      /* significand precision in bits, implicit bit included */
  int emin;   /* exponent of the smallest normal number               */
  int emax;   /* exponent of the largest finite binade                 */
  int bias;   /* exponent bias of the encoding                         */
  int mbits;  /* stored mantissa bits (p - 1)                          */
  int ebits;  /* stored exponent bits                                  */
} fmt_t;

static const fmt_t FMT_BF16 = {8, -126, 127, 127, 7, 8};
static const fmt_t FMT_F16 = {11, -14, 15, 15, 10, 5};
static const fmt_t FMT_F32 = {24, -126, 127, 127, 23, 8};

static int bit_length(uint64_t v) {
  int n = 0;
  while (v) { n++; v >>= 1; }
  return n;
}

static uint32_t encode_rounded(int neg, uint64_t sig, int e, const fmt_t* f) {
  const uint32_t sbit = (uint32_t)neg << (f->mbits + f->ebits);
  const uint32_t inf = ((1u << f->ebits) - 1u) << f->mbits;
  if (sig == 0) return sbit;
  const int E = e + bit_length(sig) - 1;                   /* 2^E <= |x| < 2^(E+1)   */
  int q = (E > f->emin ? E : f->emin) - (f->p - 1);        /* weight of the last kept bit */
  const int shift = q - e;
  uint64_t kept;
  if (shift <= 0) {
    kept = sig << (-shift);                                 /* exact, fewer than p bits */
  } else if (shift >= 64) {
    kept = 0;                                               /* |x| < half a quantum    */
  } else {
    kept = sig >> shift;
    const uint64_t rem = sig & ((1ull << shift) - 1ull);
    const uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (kept & 1ull))) kept += 1;
  }
  if (kept == (1ull << f->p)) { kept >>= 1; q += 1; }       /* carry into next binade  */
  if (kept >= (1ull << (f->p - 1))) {                       /* normal number           */
    const int Ek = q + f->p - 1;
    if (Ek > f->emax) return sbit | inf;
    return sbit | ((uint32_t)(Ek + f->bias) << f->mbits) | (uint32_t)(kept - (1ull << (f->p - 1)));
  }
  return sbit | (uint32_t)kept;                             /* subnormal               */
}

static uint32_t quiet_nan(int neg, const fmt_t* f) {
  return ((uint32_t)neg << (f->mbits + f->ebits)) | (((1u << f->ebits) - 1u) << f->mbits) |
         (1u << (f->mbits - 1));
}

static uint32_t from_f32(float x, const fmt_t* f) {
  uint32_t u;
  memcpy(&u, &x, 4);
  const int neg = (int)(u >> 31);
  const uint32_t ex = (u >> 23) & 0xFFu, man = u & 0x7FFFFFu;
  if (ex == 0xFFu) return man ? quiet_nan(neg, f) : (((uint32_t)neg << (f->mbits + f->ebits)) | (((1u << f->ebits) - 1u) << f->mbits));
  if (ex == 0) return encode_rounded(neg, man, -149, f);
  return encode_rounded(neg, (uint64_t)man | 0x800000u, (int)ex - 150, f);
}

static uint32_t from_f64(double x, const fmt_t* f) {
  uint64_t u;
  memcpy(&u, &x, 8);
  const int neg = (int)(u >> 63);
  const uint64_t ex = (u >> 52) & 0x7FFull, man = u & ((1ull << 52) - 1ull);
  if (ex == 0x7FFull) return man ? quiet_nan(neg, f) : (((uint32_t)neg << (f->mbits + f->ebits)) | (((1u << f->ebits) - 1u) << f->mbits));
  if (ex == 0) return encode_rounded(neg, man, -1074, f);
  return encode_rounded(neg, man | (1ull << 52), (int)ex - 1075, f);
}

uint16_t orc_f32_to_bf16(float f) { return (uint16_t)from_f32(f, &FMT_BF16); }
uint16_t orc_f32_to_f16(float f) { return (uint16_t)from_f32(f, &FMT_F16); }
uint16_t orc_f64_to_bf16(double d) { return (uint16_t)from_f64(d, &FMT_BF16); }
uint16_t orc_f64_to_f16(double d) { return (uint16_t)from_f64(d, &FMT_F16); }
float orc_f64_to_f32(double d) {
  const uint32_t b = from_f64(d, &FMT_F32);
  float f;
  memcpy(&f, &b, 4);
  return f;
}

/* bf16 is the high half of a binary32: widening appends 16 zero bits. */
float orc_bf16_to_f32(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* binary16 -> binary32 is exact: rebias the exponent, widen the mantissa. */
float orc_f16_to_f32(uint16_t h) {
  const int neg = h >> 15;
  const int ex = (h >> 10) & 0x1F;
  const int man = h & 0x3FF;
  float v;
  if (ex == 0x1F) {
    const uint32_t u = ((uint32_t)neg << 31) | 0x7F800000u | ((uint32_t)man << 13);
    memcpy(&v, &u, 4);
    return v;
  }
  if (ex == 0) v = ldexpf((float)man, -24);                 /* subnormal: man * 2^-24 */
  else v = ldexpf((float)(1024 + man), ex - 25);            /* (1.man) * 2^(ex-15)    */
  return neg ? -v : v;
}

int orc_elem_size(int dtype) { return dtype == ORC_FP32 ? 4 : 2; }

static double load_kind(const uint8_t* p, int kind, int64_t i) {
  switch (kind) {
    case 0: return (double)orc_bf16_to_f32(ld16(p + 2 * i));
    case 1: return (double)orc_f16_to_f32(ld16(p + 2 * i));
    case 2: {
      const uint32_t u = ld32(p + 4 * i);
      float f;
      memcpy(&f, &u, 4);
      return (double)f;
    }
    default: {
      const uint64_t u = ld64(p + 8 * i);
      double d;
      memcpy(&d, &u, 8);
      return d;
    }
  }
}

void orc_convert(const void* src, int src_kind, void* dst, int dst_kind, int64_t n) {
  const uint8_t* s = (const uint8_t*)src;
  uint8_t* d = (uint8_t*)dst;
  for (int64_t i = 0; i < n; i++) {
    if (src_kind == dst_kind) {
      const int es = src_kind == 3 ? 8 : (src_kind == 2 ? 4 : 2);
      memcpy(d + es * i, s + es * i, (size_t)es);
      continue;
    }
    const double v = load_kind(s, src_kind, i);  /* exact widening to double */
    switch (dst_kind) {
      case 0: st16(d + 2 * i, src_kind == 2 ? orc_f32_to_bf16((float)v) : orc_f64_to_bf16(v)); break;
      case 1: st16(d + 2 * i, src_kind == 2 ? orc_f32_to_f16((float)v) : orc_f64_to_f16(v)); break;
      case 2: {
        const float f = orc_f64_to_f32(v);
        uint32_t u;
        memcpy(&u, &f, 4);
        st32(d + 4 * i, u);
        break;
      }
      default: {
        uint64_t u;
        memcpy(&u, &v, 8);
        st64(d + 8 * i, u);
      }
    }
  }
}

static float load_elem(const uint8_t* p, int dtype) {
  switch (dtype) {
    case ORC_BF16: return orc_bf16_to_f32(ld16(p));
    case ORC_FP16: return orc_f16_to_f32(ld16(p));
    default: {
      const uint32_t u = ld32(p);
      float f;
      memcpy(&f, &u, 4);
      return f;
    }
  }
}

static void store_from_f32(uint8_t* p, int dtype, float v) {
  switch (dtype) {
    case ORC_BF16: st16(p, orc_f32_to_bf16(v)); break;
    case ORC_FP16: st16(p, orc_f32_to_f16(v)); break;
    default: {
      uint32_t u;
      memcpy(&u, &v, 4);
      st32(p, u);
    }
  }
}

static void store_from_f64(uint8_t* p, int dtype, double v) {
  switch (dtype) {
    case ORC_BF16: st16(p, orc_f64_to_bf16(v)); break;
    case ORC_FP16: st16(p, orc_f64_to_f16(v)); break;
    default: st32(p, from_f64(v, &FMT_F32));
  }
}

/* ------------------------------------------------------------------------ */
/* P1 "1stage：kernel 全文与时间线" (packed_reduce) and P3 "4. 求和":        */
/* widen rank 0's element to fp32, add ranks 1..W-1 in rank order in fp32,  */
/* round once to the element type.  The accumulator starts at x_0 (P1's     */
/* kernel), not at +0 (P3's pseudocode); the two differ only when every     */
/* term is -0.                                                              */
/* ------------------------------------------------------------------------ */
static float rank_sum_f32(int W, const void* const* x, int dtype, int64_t i) {
  const int es = orc_elem_size(dtype);
  float acc = load_elem((const uint8_t*)x[0] + i * es, dtype);
  for (int r = 1; r < W; r++) acc = acc + load_elem((const uint8_t*)x[r] + i * es, dtype);
  return acc;
}

void orc_reduce(int W, const void* const* x, int dtype, int64_t n, void* ar) {
  const int es = orc_elem_size(dtype);
  for (int64_t i = 0; i < n; i++) store_from_f32((uint8_t*)ar + i * es, dtype, rank_sum_f32(W, x, dtype, i));
}

/* ------------------------------------------------------------------------ */
/* P1 "2stage：分片、轮转、以及为什么没有出口 barrier": stage 1 gives rank s  */
/* the units [s*part, (s+1)*part) (the last rank up to the end) and rank s   */
/* reads the ranks starting from itself, (s + i) % W.  All ranks then gather */
/* the owner's result, so every element carries its owner's rounding.        */
/* ------------------------------------------------------------------------ */
void orc_reduce_two_shot(int W, const void* const* x, int dtype, int64_t n, void* ar) {
  const int es = orc_elem_size(dtype);
  if ((n * es) % 16 != 0) return;
  const int64_t units = n * es / 16;
  const int64_t per_unit = 16 / es;
  const int64_t part = units / W;
  for (int64_t i = 0; i < n; i++) {
    const int64_t unit = i / per_unit;
    int64_t owner = part == 0 ? W - 1 : unit / part;
    if (owner > W - 1) owner = W - 1;  /* the last rank takes the remainder */
    float acc = load_elem((const uint8_t*)x[owner] + i * es, dtype);
    for (int k = 1; k < W; k++) {
      const int r = (int)((owner + k) % W);
      acc = acc + load_elem((const uint8_t*)x[r] + i * es, dtype);
    }
    store_from_f32((uint8_t*)ar + i * es, dtype, acc);
  }
}

/* ------------------------------------------------------------------------ */
/* P4 "这个算子在算什么":                                                     */
/*   ar = sum over ranks of x;  h = ar + residual  (-> residual_out)        */
/*   rms = rsqrt(mean(h^2) + eps);  out = (h * rms) * weight (-> norm_out)   */
/* h is formed from the unrounded fp32 sum (P4 "总体设计": fp32 sum, then   */
/* add residual).  mean, rsqrt and the two products are taken in double     */
/* and rounded once to the element type.                                    */
/* ------------------------------------------------------------------------ */
void orc_reduce_residual_rmsnorm(int W, const void* const* x, const void* residual,
                                 const void* weight, float eps, int64_t M, int64_t N,
                                 int dtype, void* ar, void* residual_out, void* norm_out,
                                 double* norm_f64) {
  const int es = orc_elem_size(dtype);
  for (int64_t m = 0; m < M; m++) {
    double ss = 0.0;
    /* pass 1: rank sum, residual add, sum of squares */
    for (int64_t j = 0; j < N; j++) {
      const int64_t i = m * N + j;
      const float acc = rank_sum_f32(W, x, dtype, i);
      const float h = acc + load_elem((const uint8_t*)residual + i * es, dtype);
      if (ar) store_from_f32((uint8_t*)ar + i * es, dtype, acc);
      store_from_f32((uint8_t*)residual_out + i * es, dtype, h);
      ss += (double)h * (double)h;
    }
    const double rms = 1.0 / sqrt(ss / (double)N + (double)eps);
    /* pass 2: normalise and scale; h is recomputed exactly as in pass 1 */
    for (int64_t j = 0; j < N; j++) {
      const int64_t i = m * N + j;
      const float acc = rank_sum_f32(W, x, dtype, i);
      const float h = acc + load_elem((const uint8_t*)residual + i * es, dtype);
      const double w = (double)load_elem((const uint8_t*)weight + j * es, dtype);
      const double out = ((double)h * rms) * w;
      if (norm_f64) norm_f64[i] = out;
      store_from_f64((uint8_t*)norm_out + i * es, dtype, out);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* LL128 (P2 "LL128 的 128-byte line", "LL128 的 warp-level ready 检查"):    */
/* the data byte stream is cut into 120-byte pieces; line k holds words     */
/* 15k..15k+14 of the stream in its first 15 uint64 slots (zero past the    */
/* end of the data) and the flag in its 16th slot.                          */
/* ------------------------------------------------------------------------ */
int64_t orc_ll128_lines(int64_t D) { return (D + 119) / 120; }
int64_t orc_ll128_wire_bytes(int64_t D) { return 128 * orc_ll128_lines(D); }
int64_t orc_ll128_data_capacity(int64_t wire_bytes) { return 120 * (wire_bytes / 128); }

void orc_ll128_encode(const void* data, int64_t D, uint64_t flag, void* wire) {
  const uint8_t* src = (const uint8_t*)data;
  uint8_t* dst = (uint8_t*)wire;
  const int64_t L = orc_ll128_lines(D);
  for (int64_t k = 0; k < L; k++) {
    uint8_t* line = dst + 128 * k;
    for (int w = 0; w < 15; w++) {
      for (int j = 0; j < 8; j++) {
        const int64_t b = 120 * k + 8 * w + j;
        line[8 * w + j] = b < D ? src[b] : 0;
      }
    }
    st64(line + 120, flag);
  }
}

/* Receiver side: a line is usable only when its flag word equals the      */
/* expected flag in every rank (P2: the flag lane compares the line's       */
/* second 8-byte word of its 16-byte chunk, i.e. word 15).  Data word w of  */
/* line k is wire word 16k + w.                                             */
int64_t orc_ll128_decode_reduce(int W, const void* const* wires, int64_t D, int dtype,
                                uint64_t expected_flag, void* ar, uint32_t* stale, int64_t cap) {
  const int es = orc_elem_size(dtype);
  const int64_t L = orc_ll128_lines(D);
  int64_t n_stale = 0;
  for (int64_t k = 0; k < L; k++) {
    int line_ok = 1;
    for (int r = 0; r < W; r++) {
      const uint64_t flag = ld64((const uint8_t*)wires[r] + 128 * k + 8 * 15);
      if (flag != expected_flag) {
        if (n_stale < cap) { stale[2 * n_stale] = (uint32_t)r; stale[2 * n_stale + 1] = (uint32_t)k; }
        n_stale++;
        line_ok = 0;
      }
    }
    const int64_t b_end = 120 * k + 120 < D ? 120 * k + 120 : D;
    for (int64_t b = 120 * k; b < b_end; b += es) {
      uint8_t* out = (uint8_t*)ar + b;
      if (!line_ok) { memset(out, 0, (size_t)es); continue; }
      const int64_t wire_off = 128 * k + (b - 120 * k);  /* word (b-120k)/8 of line k */
      float acc = load_elem((const uint8_t*)wires[0] + wire_off, dtype);
      for (int r = 1; r < W; r++) acc = acc + load_elem((const uint8_t*)wires[r] + wire_off, dtype);
      store_from_f32(out, dtype, acc);
    }
  }
  return n_stale;
}

/* ------------------------------------------------------------------------ */
/* LL (P2 "LL 的 16-byte FIFO line", "LL 如何发布和等待 flag"): line i is    */
/* {data1 = low 32 bits of data word i, flag1, data2 = high 32 bits, flag2} */
/* and decodes as data1 + (data2 << 32).  A line is valid only when both    */
/* flags equal the expected flag.                                           */
/* ------------------------------------------------------------------------ */
int64_t orc_ll_lines(int64_t D) { return (D + 7) / 8; }
int64_t orc_ll_wire_bytes(int64_t D) { return 16 * orc_ll_lines(D); }
int64_t orc_ll_data_capacity(int64_t wire_bytes) { return 8 * (wire_bytes / 16); }

void orc_ll_encode(const void* data, int64_t D, uint32_t flag, void* wire) {
  const uint8_t* src = (const uint8_t*)data;
  uint8_t* dst = (uint8_t*)wire;
  const int64_t L = orc_ll_lines(D);
  for (int64_t i = 0; i < L; i++) {
    uint8_t word[8];
    for (int j = 0; j < 8; j++) word[j] = 8 * i + j < D ? src[8 * i + j] : 0;
    const uint64_t d = ld64(word);
    uint8_t* line = dst + 16 * i;
    st32(line + 0, (uint32_t)d);          /* data1 */
    st32(line + 4, flag);                 /* flag1 */
    st32(line + 8, (uint32_t)(d >> 32));  /* data2 */
    st32(line + 12, flag);                /* flag2 */
  }
}

int64_t orc_ll_decode_reduce(int W, const void* const* wires, int64_t D, int dtype,
                             uint32_t expected_flag, void* ar, uint32_t* stale, int64_t cap) {
  const int es = orc_elem_size(dtype);
  const int64_t L = orc_ll_lines(D);
  int64_t n_stale = 0;
  for (int64_t i = 0; i < L; i++) {
    int line_ok = 1;
    uint8_t words[16][8];  /* decoded data word of line i, per rank (W <= 16) */
    for (int r = 0; r < W; r++) {
      const uint8_t* line = (const uint8_t*)wires[r] + 16 * i;
      const uint32_t data1 = ld32(line), flag1 = ld32(line + 4);
      const uint32_t data2 = ld32(line + 8), flag2 = ld32(line + 12);
      if (flag1 != expected_flag || flag2 != expected_flag) {
        if (n_stale < cap) { stale[2 * n_stale] = (uint32_t)r; stale[2 * n_stale + 1] = (uint32_t)i; }
        n_stale++;
        line_ok = 0;
      }
      st64(words[r], (uint64_t)data1 + ((uint64_t)data2 << 32));
    }
    const int64_t b_end = 8 * i + 8 < D ? 8 * i + 8 : D;
    for (int64_t b = 8 * i; b < b_end; b += es) {
      uint8_t* out = (uint8_t*)ar + b;
      if (!line_ok) { memset(out, 0, (size_t)es); continue; }
      const int64_t j = b - 8 * i;
      float acc = load_elem(words[0] + j, dtype);
      for (int r = 1; r < W; r++) acc = acc + load_elem(words[r] + j, dtype);
      store_from_f32(out, dtype, acc);
    }
  }
  return n_stale;
}

/* ------------------------------------------------------------------------ */
/* Lamport one-shot push, P4 "方案二：Lamport（负零轮询）": two bf16 share a  */
/* 32-bit word (the low half holds the even element), the buffer starts as   */
/* sentinel words 0x80008000, senders turn -0.0 into +0.0 so no real word is */
/* the sentinel, and a receiver reads words until none is the sentinel.      */
/* Region = round % 3; the receive step refills another region for reuse.    */
/* ------------------------------------------------------------------------ */
void orc_lamport_fill(void* words, int64_t n_words) {
  for (int64_t i = 0; i < n_words; i++) st32((uint8_t*)words + 4 * i, ORC_LAMPORT_SENTINEL);
}

void orc_lamport_push(const void* data, int64_t n, void* slot) {
  for (int64_t i = 0; i < n; i++) {
    uint16_t v = ld16((const uint8_t*)data + 2 * i);
    if (v == 0x8000u) v = 0;  /* scrub -0.0 */
    st16((uint8_t*)slot + 2 * i, v);
  }
}

int64_t orc_lamport_reduce_residual_rmsnorm(int W, void* buffer, uint64_t round, int64_t M, int64_t N,
                                            const void* residual, const void* weight, float eps,
                                            void* ar, void* residual_out, void* norm_out,
                                            uint32_t* stale, int64_t cap) {
  const int64_t n = M * N;
  uint8_t* base = (uint8_t*)buffer;
  const int64_t region_bytes = (int64_t)W * n * 2;
  const uint8_t* region = base + (int64_t)(round % 3) * region_bytes;
  const void* x[16];
  for (int r = 0; r < W; r++) x[r] = region + (int64_t)r * n * 2;
  int64_t n_stale = 0;
  for (int64_t m = 0; m < M; m++) {
    /* a row is usable only when no word of it is the sentinel in any rank */
    int row_ok = 1;
    for (int r = 0; r < W; r++) {
      int missing = 0;
      for (int64_t j = 0; j < N; j += 2) {
        if (ld32((const uint8_t*)x[r] + 2 * (m * N + j)) == ORC_LAMPORT_SENTINEL) { missing = 1; break; }
      }
      if (missing) {
        if (n_stale < cap) { stale[2 * n_stale] = (uint32_t)r; stale[2 * n_stale + 1] = (uint32_t)m; }
        n_stale++;
        row_ok = 0;
      }
    }
    if (!row_ok) {
      memset((uint8_t*)residual_out + 2 * m * N, 0, (size_t)(2 * N));
      memset((uint8_t*)norm_out + 2 * m * N, 0, (size_t)(2 * N));
      if (ar) memset((uint8_t*)ar + 2 * m * N, 0, (size_t)(2 * N));
      continue;
    }
    const void* xr[16];
    for (int r = 0; r < W; r++) xr[r] = (const uint8_t*)x[r] + 2 * m * N;
    orc_reduce_residual_rmsnorm(W, xr, (const uint8_t*)residual + 2 * m * N, weight, eps, 1, N, ORC_BF16,
                                ar ? (uint8_t*)ar + 2 * m * N : 0, (uint8_t*)residual_out + 2 * m * N,
                                (uint8_t*)norm_out + 2 * m * N, 0);
  }
  /* refill the previous round's region so that it can take round + 2 */
  orc_lamport_fill(base + (int64_t)((round + 2) % 3) * region_bytes, region_bytes / 4);
  return n_stale;
}
