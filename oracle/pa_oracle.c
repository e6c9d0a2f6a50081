/*
 * pa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of attention over a paged
 * KV cache, in fp64.  It exists to check the CUDA library, never to serve
 * it: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (web pages on paged KV caches; cited by page and section):
 *   [SKILL] cannbot-skills "model-infer-kvcache" skill page (devpress.csdn.net)
 *           §3.1 physical layout and logical mapping, §3.3 slot_mapping,
 *           §3.6 data-flow overview, App. C sparse_mode / masks.
 *   [VLLM]  "vLLM on CANN" page (lnwmold.com): the PagedKVCache class and its
 *           read_kv gather.
 *   [MHPQ]  "Paged KV Cache and Packed Sequence in cann-recipes-infer"
 *           (mhpq.cn) §3.3: ops.paged_attention parameters, all-zero
 *           context_lengths give an all-zero output.
 *   [ATB]   "Ascend CANN ATB KV Cache and PagedAttention" (coreui.cn): the
 *           page pool, and copy-on-write of a shared page before an append.
 *
 * What it computes, in the pages' order:
 *   write  : for each new token t with slot s >= 0, the row of the pool at
 *            physical block s / block_size, offset s % block_size receives
 *            the token's K (and V) row, bit for bit   ([SKILL] §3.1, §3.3).
 *   copy   : copy-on-write of whole blocks, source to destination, in
 *            both pools ([ATB] page update race).
 *   8-bit pools: INT8 or FP8 (E4M3) codes with one scale per KV head for K
 *            and for V; the write quantises, the gather dequantises
 *            ([SKILL] App. A lists the dequantisation scales).
 *   gather : for sequence b and logical position j < L_b the key/value row
 *            is pool[block_table[b][j / block_size]][j % block_size]
 *            ([SKILL] §3.1; [VLLM] read_kv), copied into contiguous arrays.
 *   attend : naive two-pass softmax attention over the gathered rows:
 *            s_j = scale * q.K_j, m = max s_j, p_j = exp(s_j - m),
 *            o = sum p_j V_j / sum p_j;  an empty key set gives o = 0
 *            ([MHPQ] §3.3).  Decode attends to all L_b keys (sparse_mode 0);
 *            prefill row i of a sequence with q_b queries and L_b keys
 *            attends to keys j <= L_b - q_b + i (causal, sparse_mode 3,
 *            aligned so the last query sees every key: [SKILL] App. C/E).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): query head h reads KV head h / (Hq / Hkv); a negative slot means
 * "no write"; the cache layout is [num_blocks, block_size, Hkv, D] with K and
 * V in separate pools ([SKILL] §3.1).
 *
 * Inputs are raw 16-bit patterns (fp16 or bf16), decoded here exactly to
 * double from the IEEE-754 binary16 / bfloat16 definitions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { PAO_F16 = 0, PAO_BF16 = 1 };
enum {
  PAO_OK = 0,
  PAO_ERR_ARG = 1,   /* inconsistent sizes / null pointers            */
  PAO_ERR_SLOT = 2,  /* a slot at or beyond num_blocks * block_size    */
  PAO_ERR_BLOCK = 3, /* a block id outside [0, num_blocks)             */
  PAO_ERR_LEN = 4,   /* a length beyond the block table's capacity,
                        or cu_seqlens not a valid prefix sum           */
  PAO_ERR_NOMEM = 5,
  PAO_ERR_SCALE = 6  /* an INT8 scale that is not a positive finite number */
};

/* ---- exact 16-bit decoders -------------------------------------------- */

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double pao_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^(1-15-10) */
  else if (e == 0x1f)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(0x400 | f), e - 25); /* (1024+f) * 2^(e-15-10) */
  return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double pao_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int f = b & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)f, -133); /* subnormal: f * 2^(1-127-7) */
  else if (e == 0xff)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(0x80 | f), e - 134); /* (128+f) * 2^(e-127-7) */
  return sign ? -v : v;
}

static double decode16(uint16_t x, int dtype) {
  return dtype == PAO_BF16 ? pao_bf16_to_double(x) : pao_f16_to_double(x);
}

/* Decode n patterns to doubles (used by the exhaustive decoder check). */
void pao_decode_array(double *out, const uint16_t *in, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) out[i] = decode16(in[i], dtype);
}

int pao_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void pao_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ---- write: new K/V rows into the pool through slot_mapping ------------ */

/* Pools are [num_blocks, block_size, hkv, d] 16-bit patterns.  New rows are
 * [n, hkv, d] with `row_stride` elements between consecutive tokens.  A
 * negative slot is skipped; an out-of-range slot is skipped and reported.
 * The copy is a bit copy, so no decoding happens here. */
int pao_write(uint16_t *k_pool, uint16_t *v_pool, const uint16_t *k_new,
              const uint16_t *v_new, int64_t row_stride,
              const int64_t *slot_mapping, int64_t n, int hkv, int d,
              int block_size, int64_t num_blocks) {
  if (!k_pool || !v_pool || (n > 0 && (!k_new || !v_new || !slot_mapping)))
    return PAO_ERR_ARG;
  if (hkv <= 0 || d <= 0 || block_size <= 0 || num_blocks < 0 || n < 0)
    return PAO_ERR_ARG;
  int status = PAO_OK;
  const int64_t row = (int64_t)hkv * d;
  for (int64_t t = 0; t < n; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * (int64_t)block_size) {
      status = PAO_ERR_SLOT;
      continue;
    }
    int64_t block = slot / block_size; /* physical block id   */
    int64_t offset = slot % block_size; /* position in block   */
    int64_t dst = (block * block_size + offset) * row;
    for (int64_t x = 0; x < row; ++x) {
      k_pool[dst + x] = k_new[t * row_stride + x];
      v_pool[dst + x] = v_new[t * row_stride + x];
    }
  }
  return status;
}

/* ---- copy_blocks: copy-on-write of whole blocks ------------------------- */

/* [ATB] "page update race" section (copy-on-write): before a request appends
 * K/V to a page it shares with other requests, a free page is taken and the
 * whole old page is copied into it.  Here the pools are raw bytes, block b of
 * a pool being bytes [b * block_bytes, (b + 1) * block_bytes).  Pairs are
 * applied in order: block block_mapping[2p + 1] of the K pool and of the V
 * pool receives block block_mapping[2p] byte for byte.  A pair naming a block
 * outside [0, num_blocks) copies nothing and is reported. */
int pao_copy_blocks(uint8_t *k_pool, uint8_t *v_pool, int64_t block_bytes,
                    int64_t num_blocks, const int64_t *block_mapping, int64_t n) {
  if (!k_pool || !v_pool || (n > 0 && !block_mapping)) return PAO_ERR_ARG;
  if (block_bytes <= 0 || num_blocks < 0 || n < 0) return PAO_ERR_ARG;
  int status = PAO_OK;
  for (int64_t p = 0; p < n; ++p) {
    const int64_t src = block_mapping[2 * p], dst = block_mapping[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      status = PAO_ERR_BLOCK;
      continue;
    }
    memmove(k_pool + dst * block_bytes, k_pool + src * block_bytes,
            (size_t)block_bytes);
    memmove(v_pool + dst * block_bytes, v_pool + src * block_bytes,
            (size_t)block_bytes);
  }
  return status;
}

/* ---- gather: one sequence's keys/values for one KV head ---------------- */

/* Fills kc, vc ([len, d] doubles) with logical positions 0..len-1 of the
 * sequence whose block-table row is `bt_row`, for KV head g. */
static int gather(double *kc, double *vc, const uint16_t *k_pool,
                  const uint16_t *v_pool, const int32_t *bt_row, int len,
                  int g, int hkv, int d, int block_size, int64_t num_blocks,
                  int dtype) {
  for (int j = 0; j < len; ++j) {
    int logical_block = j / block_size;
    int offset = j % block_size;
    int32_t block = bt_row[logical_block];
    if (block < 0 || block >= num_blocks) return PAO_ERR_BLOCK;
    int64_t base = (((int64_t)block * block_size + offset) * hkv + g) * d;
    for (int x = 0; x < d; ++x) {
      kc[(int64_t)j * d + x] = decode16(k_pool[base + x], dtype);
      vc[(int64_t)j * d + x] = decode16(v_pool[base + x], dtype);
    }
  }
  return PAO_OK;
}

/* ---- INT8 pool: per-KV-head symmetric quantisation --------------------- */

/* [SKILL] App. A lists the fused operator's quantised-KV parameters (one
 * dequantisation scale for the key and one for the value) and the page's
 * "advanced features" note names an INT8 KV cache; neither prints the
 * formula.  Reading taken: one fp32 scale per KV head for K and one for V,
 * codes in [-127, 127], code = round-half-to-even(x / scale) with the
 * division and the rounding done in fp32 (IEEE, round to nearest -- the
 * precision the kernels decide the code in), a NaN input gives code 0, and
 * the dequantised value is code * scale. */
static int scale_ok(float s) { return s > 0.0f && s <= 3.4028234663852886e38f; }

static int8_t quantize1(float x, float scale) {
  if (x != x) return 0;
  float y = x / scale;
  if (y >= 127.0f) return 127;
  if (y <= -127.0f) return -127;
  return (int8_t)rintf(y);
}

/* Codes of n 16-bit values under one scale (all 0 for a bad scale). */
int pao_quantize_int8(int8_t *codes, const uint16_t *x, int64_t n, int dtype,
                      float scale) {
  if (!codes || (n > 0 && !x) || n < 0) return PAO_ERR_ARG;
  const int good = scale_ok(scale);
  for (int64_t i = 0; i < n; ++i)
    codes[i] = good ? quantize1((float)decode16(x[i], dtype), scale) : 0;
  return good ? PAO_OK : PAO_ERR_SCALE;
}

/* The write of pao_write into INT8 pools: each new row is quantised per KV
 * head g with k_scale[g] / v_scale[g]. */
int pao_write_int8(int8_t *k_pool, int8_t *v_pool, const uint16_t *k_new,
                   const uint16_t *v_new, int64_t row_stride,
                   const int64_t *slot_mapping, int64_t n, int hkv, int d,
                   int block_size, int64_t num_blocks, int dtype,
                   const float *k_scale, const float *v_scale) {
  if (!k_pool || !v_pool || !k_scale || !v_scale ||
      (n > 0 && (!k_new || !v_new || !slot_mapping)))
    return PAO_ERR_ARG;
  if (hkv <= 0 || d <= 0 || block_size <= 0 || num_blocks < 0 || n < 0)
    return PAO_ERR_ARG;
  int status = PAO_OK;
  for (int g = 0; g < hkv; ++g)
    if (!scale_ok(k_scale[g]) || !scale_ok(v_scale[g])) status = PAO_ERR_SCALE;
  const int64_t row = (int64_t)hkv * d;
  for (int64_t t = 0; t < n; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * (int64_t)block_size) {
      status = PAO_ERR_SLOT;
      continue;
    }
    int64_t block = slot / block_size, offset = slot % block_size;
    int64_t dst = (block * block_size + offset) * row;
    for (int g = 0; g < hkv; ++g) {
      const float ks = k_scale[g], vs = v_scale[g];
      const int good = scale_ok(ks) && scale_ok(vs);
      for (int x = 0; x < d; ++x) {
        int64_t i = (int64_t)g * d + x;
        k_pool[dst + i] = good ? quantize1((float)decode16(k_new[t * row_stride + i], dtype), ks) : 0;
        v_pool[dst + i] = good ? quantize1((float)decode16(v_new[t * row_stride + i], dtype), vs) : 0;
      }
    }
  }
  return status;
}

/* ---- FP8 (E4M3) pools ---------------------------------------------------- */

/* The value of an E4M3 code: 1 sign bit, 4 exponent bits (bias 7), 3
 * fraction bits; exponent field 0 is subnormal (f / 8 * 2^-6); S.1111.111 is
 * NaN; there are no infinities, so the largest finite value is 448. */
static double e4m3_value(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp(m / 8.0, -6);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

void pao_fp8_value(double *out, const uint8_t *codes, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

/* The E4M3 code nearest to y (ties to the even code), saturating to the
 * largest finite value; the sign bit follows y's (so -0 and negative values
 * that round to zero give 0x80).  Finite magnitudes grow with the code
 * (0x00 .. 0x7E), so bisection finds the two codes around |y| and the nearer
 * one wins. */
static uint8_t e4m3_nearest(float y) {
  const uint8_t sign = signbit(y) ? 0x80 : 0x00;
  const double a = fabs((double)y);
  if (!(a < 448.0)) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 0x7E; /* value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (e4m3_value((uint8_t)mid) <= a) lo = mid;
    else hi = mid;
  }
  const double dl = a - e4m3_value((uint8_t)lo), dh = e4m3_value((uint8_t)hi) - a;
  const int best = dl < dh ? lo : (dh < dl ? hi : ((lo & 1) == 0 ? lo : hi));
  return (uint8_t)(sign | best);
}

/* An FP8 code of x under `scale`: the nearest E4M3 value to x / scale, the
 * division in fp32; a NaN input is stored as code 0. */
static uint8_t quantize_fp8_1(float x, float scale) {
  if (x != x) return 0;
  return e4m3_nearest(x / scale);
}

int pao_quantize_fp8(uint8_t *codes, const uint16_t *x, int64_t n, int dtype,
                     float scale) {
  if (!codes || (n > 0 && !x) || n < 0) return PAO_ERR_ARG;
  const int good = scale_ok(scale);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    codes[i] = good ? quantize_fp8_1((float)decode16(x[i], dtype), scale) : 0;
  return good ? PAO_OK : PAO_ERR_SCALE;
}

/* The write of pao_write into FP8 pools, quantised per KV head g with
 * k_scale[g] / v_scale[g] (a head with a bad scale stores code 0). */
int pao_write_fp8(uint8_t *k_pool, uint8_t *v_pool, const uint16_t *k_new,
                  const uint16_t *v_new, int64_t row_stride,
                  const int64_t *slot_mapping, int64_t n, int hkv, int d,
                  int block_size, int64_t num_blocks, int dtype,
                  const float *k_scale, const float *v_scale) {
  if (!k_pool || !v_pool || !k_scale || !v_scale ||
      (n > 0 && (!k_new || !v_new || !slot_mapping)))
    return PAO_ERR_ARG;
  if (hkv <= 0 || d <= 0 || block_size <= 0 || num_blocks < 0 || n < 0)
    return PAO_ERR_ARG;
  int status = PAO_OK;
  for (int g = 0; g < hkv; ++g)
    if (!scale_ok(k_scale[g]) || !scale_ok(v_scale[g])) status = PAO_ERR_SCALE;
  const int64_t row = (int64_t)hkv * d;
  for (int64_t t = 0; t < n; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * (int64_t)block_size) {
      status = PAO_ERR_SLOT;
      continue;
    }
    const int64_t dst = ((slot / block_size) * block_size + slot % block_size) * row;
    for (int g = 0; g < hkv; ++g) {
      const float fks = k_scale[g], fvs = v_scale[g];
      const int good = scale_ok(fks) && scale_ok(fvs);
      for (int x = 0; x < d; ++x) {
        const int64_t i = (int64_t)g * d + x;
        const float kx = (float)decode16(k_new[t * row_stride + i], dtype);
        const float vx = (float)decode16(v_new[t * row_stride + i], dtype);
        k_pool[dst + i] = good ? quantize_fp8_1(kx, fks) : 0;
        v_pool[dst + i] = good ? quantize_fp8_1(vx, fvs) : 0;
      }
    }
  }
  return status;
}

/* gather from FP8 pools: the rows dequantised with KV head g's scales. */
static int gather_fp8(double *kc, double *vc, const uint8_t *k_pool,
                      const uint8_t *v_pool, const int32_t *bt_row, int len,
                      int g, int hkv, int d, int block_size, int64_t num_blocks,
                      double k_scale, double v_scale) {
  double value[256]; /* every code's value, once per call */
  for (int c = 0; c < 256; ++c) value[c] = e4m3_value((uint8_t)c);
  for (int j = 0; j < len; ++j) {
    int32_t block = bt_row[j / block_size];
    if (block < 0 || block >= num_blocks) return PAO_ERR_BLOCK;
    int64_t base = (((int64_t)block * block_size + j % block_size) * hkv + g) * d;
    for (int x = 0; x < d; ++x) {
      kc[(int64_t)j * d + x] = value[k_pool[base + x]] * k_scale;
      vc[(int64_t)j * d + x] = value[v_pool[base + x]] * v_scale;
    }
  }
  return PAO_OK;
}

/* gather from INT8 pools: the rows dequantised with KV head g's scales. */
static int gather_int8(double *kc, double *vc, const int8_t *k_pool,
                       const int8_t *v_pool, const int32_t *bt_row, int len,
                       int g, int hkv, int d, int block_size, int64_t num_blocks,
                       double k_scale, double v_scale) {
  for (int j = 0; j < len; ++j) {
    int32_t block = bt_row[j / block_size];
    if (block < 0 || block >= num_blocks) return PAO_ERR_BLOCK;
    int64_t base = (((int64_t)block * block_size + j % block_size) * hkv + g) * d;
    for (int x = 0; x < d; ++x) {
      kc[(int64_t)j * d + x] = (double)k_pool[base + x] * k_scale;
      vc[(int64_t)j * d + x] = (double)v_pool[base + x] * v_scale;
    }
  }
  return PAO_OK;
}

/* ---- attend: naive two-pass softmax attention for one query row -------- */

/* o[d] = sum_j softmax(scale * q.K_j) V_j over keys 0..n-1; o = 0 if n <= 0.
 * `s` is caller scratch of at least n doubles. */
static void attend(double *o, const double *q, const double *kc,
                   const double *vc, int n, int d, double scale, double *s) {
  if (n <= 0) {
    for (int x = 0; x < d; ++x) o[x] = 0.0;
    return;
  }
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int x = 0; x < d; ++x) dot += q[x] * kc[(int64_t)j * d + x];
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  double denom = 0.0;
  for (int j = 0; j < n; ++j) {
    s[j] = exp(s[j] - m);
    denom += s[j];
  }
  for (int x = 0; x < d; ++x) {
    double acc = 0.0;
    for (int j = 0; j < n; ++j) acc += s[j] * vc[(int64_t)j * d + x];
    o[x] = acc / denom;
  }
}

/* ---- decode: one query token per sequence ------------------------------ */

/* q: [num_seqs, hq, d] patterns with q_row_stride elements between
 * sequences (heads contiguous).  out: [num_seqs, hq, d] doubles.
 * block_table: [num_seqs, bt_stride] int32 of which the first
 * max_blocks_per_seq columns may be used.  context_lens: [num_seqs]. */
/* Pools of 16-bit patterns (k_scale == NULL), or INT8 codes (fp8 == 0) or
 * FP8 E4M3 codes (fp8 != 0) with per-KV-head scales k_scale / v_scale. */
static int decode_common(double *out, const uint16_t *q, int64_t q_row_stride,
                         const void *k_pool, const void *v_pool,
                         const int32_t *block_table, int64_t bt_stride,
                         int max_blocks_per_seq, const int32_t *context_lens,
                         int num_seqs, int hq, int hkv, int d, int block_size,
                         int64_t num_blocks, double scale, int dtype,
                         const float *k_scale, const float *v_scale, int fp8) {
  if (!out || !q || !k_pool || !v_pool || !block_table || !context_lens)
    return PAO_ERR_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || block_size <= 0)
    return PAO_ERR_ARG;
  const int group = hq / hkv;
  int status = PAO_OK;
  const int units = num_seqs * hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int u = 0; u < units; ++u) {
    int b = u / hkv, g = u % hkv;
    int len = context_lens[b];
    int err = PAO_OK;
    if (len < 0 || (int64_t)len > (int64_t)max_blocks_per_seq * block_size)
      err = PAO_ERR_LEN;
    double *kc = NULL, *vc = NULL, *s = NULL, *qd = NULL;
    if (err == PAO_OK) {
      size_t rows = len > 0 ? (size_t)len : 1;
      kc = (double *)malloc(rows * d * sizeof(double));
      vc = (double *)malloc(rows * d * sizeof(double));
      s = (double *)malloc(rows * sizeof(double));
      qd = (double *)malloc((size_t)d * sizeof(double));
      if (!kc || !vc || !s || !qd) err = PAO_ERR_NOMEM;
    }
    if (err == PAO_OK && k_scale && fp8)
      err = gather_fp8(kc, vc, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                       block_table + (int64_t)b * bt_stride, len, g, hkv, d,
                       block_size, num_blocks, k_scale[g], v_scale[g]);
    else if (err == PAO_OK && k_scale)
      err = gather_int8(kc, vc, (const int8_t *)k_pool, (const int8_t *)v_pool,
                        block_table + (int64_t)b * bt_stride, len, g, hkv, d,
                        block_size, num_blocks, k_scale[g], v_scale[g]);
    else if (err == PAO_OK)
      err = gather(kc, vc, (const uint16_t *)k_pool, (const uint16_t *)v_pool,
                   block_table + (int64_t)b * bt_stride, len, g, hkv, d,
                   block_size, num_blocks, dtype);
    for (int h = g * group; h < (g + 1) * group; ++h) {
      double *o = out + ((int64_t)b * hq + h) * d;
      if (err != PAO_OK) {
        for (int x = 0; x < d; ++x) o[x] = NAN;
        continue;
      }
      for (int x = 0; x < d; ++x)
        qd[x] = decode16(q[(int64_t)b * q_row_stride + (int64_t)h * d + x], dtype);
      attend(o, qd, kc, vc, len, d, scale, s);
    }
    free(kc);
    free(vc);
    free(s);
    free(qd);
    if (err != PAO_OK) {
#pragma omp critical
      status = err;
    }
  }
  return status;
}

int pao_decode(double *out, const uint16_t *q, int64_t q_row_stride,
               const uint16_t *k_pool, const uint16_t *v_pool,
               const int32_t *block_table, int64_t bt_stride,
               int max_blocks_per_seq, const int32_t *context_lens,
               int num_seqs, int hq, int hkv, int d, int block_size,
               int64_t num_blocks, double scale, int dtype) {
  return decode_common(out, q, q_row_stride, k_pool, v_pool, block_table,
                       bt_stride, max_blocks_per_seq, context_lens, num_seqs,
                       hq, hkv, d, block_size, num_blocks, scale, dtype, NULL,
                       NULL, 0);
}

/* Decode over INT8 pools, dequantised per KV head (see pao_write_int8). */
int pao_decode_int8(double *out, const uint16_t *q, int64_t q_row_stride,
                    const int8_t *k_pool, const int8_t *v_pool,
                    const int32_t *block_table, int64_t bt_stride,
                    int max_blocks_per_seq, const int32_t *context_lens,
                    int num_seqs, int hq, int hkv, int d, int block_size,
                    int64_t num_blocks, double scale, int dtype,
                    const float *k_scale, const float *v_scale) {
  if (!k_scale || !v_scale) return PAO_ERR_ARG;
  return decode_common(out, q, q_row_stride, k_pool, v_pool, block_table,
                       bt_stride, max_blocks_per_seq, context_lens, num_seqs,
                       hq, hkv, d, block_size, num_blocks, scale, dtype, k_scale,
                       v_scale, 0);
}

/* Decode over FP8 (E4M3) pools, dequantised per KV head (see pao_write_fp8). */
int pao_decode_fp8(double *out, const uint16_t *q, int64_t q_row_stride,
                   const uint8_t *k_pool, const uint8_t *v_pool,
                   const int32_t *block_table, int64_t bt_stride,
                   int max_blocks_per_seq, const int32_t *context_lens,
                   int num_seqs, int hq, int hkv, int d, int block_size,
                   int64_t num_blocks, double scale, int dtype,
                   const float *k_scale, const float *v_scale) {
  if (!k_scale || !v_scale) return PAO_ERR_ARG;
  return decode_common(out, q, q_row_stride, k_pool, v_pool, block_table,
                       bt_stride, max_blocks_per_seq, context_lens, num_seqs,
                       hq, hkv, d, block_size, num_blocks, scale, dtype, k_scale,
                       v_scale, 1);
}

/* ---- prefill: packed variable-length queries --------------------------- */

/* q: [total_q, hq, d] patterns, sequence b owning rows cu_seqlens_q[b] ..
 * cu_seqlens_q[b+1]-1.  context_lens[b] = L_b keys in the cache.  With
 * `causal`, row i of sequence b attends keys 0 .. L_b - q_b + i; otherwise
 * all L_b keys.  If `row_mask` is non-null only rows t with row_mask[t] != 0
 * are computed (the others are left untouched).  out: [total_q, hq, d]. */
int pao_prefill(double *out, const uint16_t *q, int64_t q_row_stride,
                const uint16_t *k_pool, const uint16_t *v_pool,
                const int32_t *block_table, int64_t bt_stride,
                int max_blocks_per_seq, const int32_t *cu_seqlens_q,
                const int32_t *context_lens, int num_seqs, int64_t total_q,
                int hq, int hkv, int d, int block_size, int64_t num_blocks,
                double scale, int causal, const uint8_t *row_mask, int dtype) {
  if (!out || !q || !k_pool || !v_pool || !block_table || !cu_seqlens_q ||
      !context_lens)
    return PAO_ERR_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || block_size <= 0)
    return PAO_ERR_ARG;
  /* cu_seqlens must be a prefix sum: starts at 0, never decreases, ends at
   * the packed total. */
  if (cu_seqlens_q[0] != 0 || cu_seqlens_q[num_seqs] != total_q)
    return PAO_ERR_LEN;
  for (int b = 0; b < num_seqs; ++b)
    if (cu_seqlens_q[b + 1] < cu_seqlens_q[b]) return PAO_ERR_LEN;
  const int group = hq / hkv;
  int status = PAO_OK;
  const int units = num_seqs * hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int u = 0; u < units; ++u) {
    int b = u / hkv, g = u % hkv;
    int len = context_lens[b];
    int first = cu_seqlens_q[b];
    int qlen = cu_seqlens_q[b + 1] - first;
    int err = PAO_OK;
    if (len < 0 || (int64_t)len > (int64_t)max_blocks_per_seq * block_size)
      err = PAO_ERR_LEN;
    int needed = 0; /* any row of this sequence requested? */
    for (int i = 0; i < qlen; ++i)
      if (!row_mask || row_mask[first + i]) needed = 1;
    if (!needed) continue;
    double *kc = NULL, *vc = NULL, *s = NULL, *qd = NULL;
    if (err == PAO_OK) {
      size_t rows = len > 0 ? (size_t)len : 1;
      kc = (double *)malloc(rows * d * sizeof(double));
      vc = (double *)malloc(rows * d * sizeof(double));
      s = (double *)malloc(rows * sizeof(double));
      qd = (double *)malloc((size_t)d * sizeof(double));
      if (!kc || !vc || !s || !qd) err = PAO_ERR_NOMEM;
    }
    if (err == PAO_OK)
      err = gather(kc, vc, k_pool, v_pool, block_table + (int64_t)b * bt_stride,
                   len, g, hkv, d, block_size, num_blocks, dtype);
    for (int i = 0; i < qlen; ++i) {
      int64_t t = first + i;
      if (row_mask && !row_mask[t]) continue;
      int n = causal ? len - qlen + i + 1 : len;
      if (n > len) n = len;
      for (int h = g * group; h < (g + 1) * group; ++h) {
        double *o = out + (t * hq + h) * d;
        if (err != PAO_OK) {
          for (int x = 0; x < d; ++x) o[x] = NAN;
          continue;
        }
        for (int x = 0; x < d; ++x)
          qd[x] = decode16(q[t * q_row_stride + (int64_t)h * d + x], dtype);
        attend(o, qd, kc, vc, n, d, scale, s);
      }
    }
    free(kc);
    free(vc);
    free(s);
    free(qd);
    if (err != PAO_OK) {
#pragma omp critical
      status = err;
    }
  }
  return status;
}
