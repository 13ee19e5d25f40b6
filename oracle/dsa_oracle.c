/*
 * dsa_oracle.c -- plain, slow, fp64 CPU oracle for paged sparse/sliding-window
 * MQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links or calls this
 * file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * load it. It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, per decode token t and query head h (the plain definition
 * of the result; no blocking, splitting or fusion):
 *
 *   1. Candidate rows.  Sources: the vLLM "swapab_decode_attn" page
 *      (SwapABDecodeKernel.stage_inputs: a slot counts only when its list
 *      position is below min(len, width), its id is non-negative and its id
 *      is below the cache's slot count) and the CuTeDSL
 *      "native_swa_decode.py" page (_fallback_batched_sdp masks positions
 *      past the length and negative ids).
 *      For each list L (sliding window, then the optional extra list) and
 *      position r in [0, width_L): limit = clamp(lens_L[t], 0, width_L); the
 *      row is kept iff r < limit and 0 <= id < num_pages*page_size with
 *      id = idx_L[t, r]. Every kept occurrence is one key/value row; both
 *      lists feed one softmax.
 *   2. Address.  block = id / page_size, offset = id % page_size; the record
 *      starts at base + block*page_stride + offset*record_bytes (swapab page,
 *      stage_inputs splits the id by the power-of-two page size; its
 *      __call__ docstring allows pages further apart than page*record).
 *   3. Dequantize in fp64 (record formats: the fp8 record holds 512 e4m3
 *      bytes then 4 little-endian fp32 scales, one per 128 dims; the V4.1
 *      fp8 record of the swapab page (stage_inputs, fp8 branch) holds 512
 *      e4m3 bytes then 16 ue8m0 scale bytes, one per 32 dims, scale byte b
 *      meaning 2^(b-127); the NVFP4 record holds 256 bytes of e2m1 nibbles
 *      then 32 e4m3 scales, one per 16 dims, element 2i in the low nibble of
 *      byte i and 2i+1 in the high one). k[d] = code(d) * scale(d).
 *      The MODEL1 record of FlashMLA's sparse_decode.h page (the check
 *      bytes_per_token = 448 + 64*2 + (448/64)*1 + 1 for d_qk = d_v = 512;
 *      the page gives only these byte counts, read here in the order they
 *      are summed): bytes 0..447 are the e4m3 codes of dims 0..447, bytes
 *      448..575 dims 448..511 as little-endian bf16 values, bytes 576..582
 *      one ue8m0 scale byte per 64 fp8 dims (dim d takes byte 576 + d/64,
 *      meaning 2^(b-127)), byte 583 unused: k[d] = e4m3(byte d) *
 *      2^(byte[576 + d/64] - 127) for d < 448, k[d] = bf16 value for
 *      d >= 448.
 *      The V3.2 record of the same page (bytes_per_token = 512 + 64*2 +
 *      (512/128)*4 for d_qk = 576, d_v = 512; again only byte counts):
 *      read as the fp8 record above (512 e4m3 codes, then 4 little-endian
 *      fp32 scales, one per 128 dims) followed by the 64 extra key dims as
 *      little-endian bf16 values (bytes 528..655). The key has 576 dims,
 *      k[d] = e4m3(byte d) * scale(d / 128) for d < 512 and k[512 + i] =
 *      bf16 value i; the value row is k[0..511]. Q then has 576 dims, taken
 *      as given (the page's kernel applies no rotation; a RoPE table is
 *      rejected with this record), and out has 512.
 *   4. Q.  q = bf16 value of q[t, h, :] in fp64. With RoPE on, the last 64
 *      dims are rotated by the fp32 table row cos_sin[positions[t]] =
 *      [cos(32) | sin(32)], pair i taking c = cos[i], s = sin[i]:
 *      NeoX style pairs x1 = q[448+i] with x2 = q[480+i]; GPT-J style (the
 *      swapab page, stage_inputs Q RoPE) pairs x1 = q[448+2i] with
 *      x2 = q[449+2i]; either way x1 <- x1 c - x2 s, x2 <- x2 c + x1 s.
 *   5. Scores s_j = scale * (q . k_j). The sink logit is not scaled
 *      (swapab page, merge step: the sink enters as exp(sink) in natural-log
 *      units next to the partial sums).
 *   6. lse = log(sum_j exp(s_j)) over the real keys only (natural log),
 *      -inf when no row is kept.
 *      out = sum_j exp(s_j) k_j / (sum_j exp(s_j) + exp(sink)); V = K (one
 *      shared row serves as key and value). No rows, or sink = +inf, gives
 *      out = 0 (swapab page, merge step: a zero denominator or an infinite
 *      sink yields a zero output).
 *
 * The V4.1 output epilogue (swapab page, merge step: inverse RoPE, MXFP8
 * cast, o-fused store) is a separate function, oracle_mxfp8_epilogue, applied
 * to the fp64 out of steps 1-6.
 *
 * Masking instrumentation: per token, the count of kept rows and the sum
 * (mod 2^32) over kept rows of fmix32(id * 0x9E3779B1 + 2*r + L), where
 * fmix32 is the MurmurHash3 32-bit finalizer. Lets a test compare row
 * selection bit-exactly without exporting masks.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_D 512      /* value dims (and key dims, but for the V3.2 record) */
#define ORACLE_DQK_V32 576
#define ORACLE_ROPE_START 448
#define ORACLE_ROPE_HALF 32

enum {
  ORACLE_FMT_FP8_528 = 0,
  ORACLE_FMT_NVFP4_288 = 1,
  ORACLE_FMT_FP8_528_UE8M0 = 2,
  ORACLE_FMT_MODEL1_584 = 3,
  ORACLE_FMT_V32_656 = 4
};
enum { ORACLE_ROPE_NEOX = 0, ORACLE_ROPE_GPTJ = 1 };

typedef struct {
  const uint8_t *base;  /* host bytes of the whole cache                      */
  int64_t num_pages;
  int64_t page_stride;  /* bytes between consecutive pages                    */
  int32_t page_size;    /* slots per page                                     */
  int32_t format;       /* ORACLE_FMT_*                                       */
} oracle_cache;

typedef struct {
  const int32_t *ids;   /* [T, row_stride] slot ids                           */
  const int32_t *lens;  /* [T]                                                */
  int64_t row_stride;   /* elements between tokens                            */
  int32_t width;
  int32_t pad_;
} oracle_list;

/* OCP FP8 E4M3 ("FN") value: 1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is
 * NaN; there is no infinity. */
double oracle_e4m3_value(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 3) & 0xF;
  int m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* OCP FP4 E2M1 value: 1 sign bit, 2 exponent bits with bias 1, 1 mantissa
 * bit; exponent field 0 is subnormal (m * 0.5). */
double oracle_e2m1_value(uint8_t nib) {
  int sign = (nib >> 3) & 1;
  int e = (nib >> 1) & 3;
  int m = nib & 1;
  double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
  return sign ? -v : v;
}

/* OCP MX E8M0 scale: 2^(b - 127); b = 0xFF is NaN. */
double oracle_ue8m0_value(uint8_t b) {
  if (b == 0xFF) return NAN;
  return ldexp(1.0, (int)b - 127);
}

static double le_f32(const uint8_t *p) {
  uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
               ((uint32_t)p[3] << 24);
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double bf16_value(uint16_t u) {
  uint32_t w = (uint32_t)u << 16;
  float f;
  memcpy(&f, &w, 4);
  return (double)f;
}

static int record_bytes(int32_t format) {
  if (format == ORACLE_FMT_NVFP4_288) return 288;
  if (format == ORACLE_FMT_V32_656) return 656;
  return format == ORACLE_FMT_MODEL1_584 ? 584 : 528;
}

/* Step 3: one record -> its key dims in fp64 (512 values; 576 for the V3.2
 * record). */
void oracle_dequant_record(const uint8_t *rec, int32_t format, double *k) {
  if (format == ORACLE_FMT_FP8_528 || format == ORACLE_FMT_V32_656) {
    for (int d = 0; d < ORACLE_D; ++d)
      k[d] = oracle_e4m3_value(rec[d]) * le_f32(rec + 512 + 4 * (d / 128));
    if (format == ORACLE_FMT_V32_656)
      for (int i = 0; i < ORACLE_DQK_V32 - ORACLE_D; ++i) {
        const uint8_t *b = rec + 528 + 2 * i;
        k[ORACLE_D + i] = bf16_value((uint16_t)(b[0] | (b[1] << 8)));
      }
  } else if (format == ORACLE_FMT_FP8_528_UE8M0) {
    for (int d = 0; d < ORACLE_D; ++d)
      k[d] = oracle_e4m3_value(rec[d]) * oracle_ue8m0_value(rec[512 + d / 32]);
  } else if (format == ORACLE_FMT_MODEL1_584) {
    for (int d = 0; d < 448; ++d)
      k[d] = oracle_e4m3_value(rec[d]) * oracle_ue8m0_value(rec[576 + d / 64]);
    for (int d = 448; d < ORACLE_D; ++d) {
      const uint8_t *b = rec + 448 + 2 * (d - 448);
      k[d] = bf16_value((uint16_t)(b[0] | (b[1] << 8)));
    }
  } else {
    for (int d = 0; d < ORACLE_D; ++d) {
      uint8_t byte = rec[d / 2];
      uint8_t nib = (d % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
      k[d] = oracle_e2m1_value(nib) * oracle_e4m3_value(rec[256 + d / 16]);
    }
  }
}

static uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

/* Step 1 for one token: kept rows of one list -> appended to K. */
static int64_t gather_list(const oracle_cache *c, const oracle_list *l, int32_t lid,
                           int32_t t, int dk, double *K, int64_t n, uint32_t *sum) {
  int32_t len = l->lens[t];
  int32_t limit = len < 0 ? 0 : (len > l->width ? l->width : len);
  int64_t slots = c->num_pages * (int64_t)c->page_size;
  int rb = record_bytes(c->format);
  for (int32_t r = 0; r < limit; ++r) {
    int32_t id = l->ids[(int64_t)t * l->row_stride + r];
    if (id < 0 || (int64_t)id >= slots) continue;
    int64_t blk = (int64_t)id / c->page_size;
    int64_t off = (int64_t)id % c->page_size;
    const uint8_t *rec = c->base + blk * c->page_stride + off * rb;
    oracle_dequant_record(rec, c->format, K + n * dk);
    *sum += fmix32((uint32_t)id * 0x9E3779B1u + 2u * (uint32_t)r + (uint32_t)lid);
    ++n;
  }
  return n;
}

typedef struct {
  int32_t H;
  const uint16_t *q;
  int64_t q_st, q_sh;
  const oracle_cache *caches;
  const oracle_list *lists;
  int32_t nlists;
  const float *sink;
  const int64_t *positions;
  const float *cos_sin;
  int64_t cs_rows;
  int32_t rope_style;   /* ORACLE_ROPE_* */
  int32_t dk;           /* key / query dims: 512, or 576 with V3.2 records */
  double scale;
  const int32_t *tokens;
  int32_t n_tokens;
  double *out;
  double *lse;
  int32_t *kept;
  uint32_t *checksum;
  int32_t nthreads;
  int32_t tid;
  int32_t status;
} oracle_job;

static void one_token(oracle_job *J, int32_t i, double *K, double *s) {
  int32_t t = J->tokens[i];
  int64_t n = 0;
  uint32_t sum = 0;
  for (int32_t L = 0; L < J->nlists; ++L)
    n = gather_list(&J->caches[L], &J->lists[L], L, t, J->dk, K, n, &sum);
  J->kept[i] = (int32_t)n;
  J->checksum[i] = sum;

  double q[ORACLE_DQK_V32];
  const int dk = J->dk;
  for (int32_t h = 0; h < J->H; ++h) {
    const uint16_t *qh = J->q + (int64_t)t * J->q_st + (int64_t)h * J->q_sh;
    for (int d = 0; d < dk; ++d) q[d] = bf16_value(qh[d]);
    if (J->cos_sin) {
      int64_t pos = J->positions[t];
      const float *row = J->cos_sin + pos * 64;
      for (int i2 = 0; i2 < ORACLE_ROPE_HALF; ++i2) {
        double c = (double)row[i2], sn = (double)row[ORACLE_ROPE_HALF + i2];
        int d1, d2;   /* the pair's two dims */
        if (J->rope_style == ORACLE_ROPE_GPTJ) {
          d1 = ORACLE_ROPE_START + 2 * i2;
          d2 = d1 + 1;
        } else {
          d1 = ORACLE_ROPE_START + i2;
          d2 = d1 + ORACLE_ROPE_HALF;
        }
        double x1 = q[d1], x2 = q[d2];
        q[d1] = x1 * c - x2 * sn;
        q[d2] = x2 * c + x1 * sn;
      }
    }
    /* Step 5: scores. */
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      const double *k = K + j * dk;
      double dot = 0.0;
      for (int d = 0; d < dk; ++d) dot += q[d] * k[d];
      s[j] = J->scale * dot;
      if (s[j] > mx) mx = s[j];
    }
    /* Step 6: lse over real keys; out with the sink in the denominator. */
    double *o = J->out + ((int64_t)i * J->H + h) * ORACLE_D;
    for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
    double *lse = J->lse + (int64_t)i * J->H + h;
    if (n == 0) {
      *lse = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) z += exp(s[j] - mx);
    *lse = mx + log(z);
    double sk = J->sink ? (double)J->sink[h] : -INFINITY;
    if (sk == INFINITY) continue; /* exp(sink) dominates: out = 0 */
    /* out = sum_j e^{s_j - mx} k_j / (z + e^{sink - mx}) */
    double den = z + exp(sk - mx);
    for (int64_t j = 0; j < n; ++j) {
      double w = exp(s[j] - mx) / den;
      const double *k = K + j * dk;   /* the value: the key's first 512 dims */
      for (int d = 0; d < ORACLE_D; ++d) o[d] += w * k[d];
    }
  }
}

static void *worker(void *arg) {
  oracle_job *J = (oracle_job *)arg;
  int64_t maxrows = 0;
  for (int32_t L = 0; L < J->nlists; ++L) maxrows += J->lists[L].width;
  double *K = (double *)malloc((size_t)(maxrows > 0 ? maxrows : 1) * J->dk * sizeof(double));
  double *s = (double *)malloc((size_t)(maxrows > 0 ? maxrows : 1) * sizeof(double));
  if (!K || !s) {
    J->status = -1;
  } else {
    for (int32_t i = J->tid; i < J->n_tokens; i += J->nthreads) one_token(J, i, K, s);
  }
  free(K);
  free(s);
  return NULL;
}

/* Runs steps 1-6 for the listed tokens. Outputs are indexed by position in
 * `tokens`: out[n_tokens][H][512], lse[n_tokens][H], kept[n_tokens],
 * checksum[n_tokens]. rope_style: ORACLE_ROPE_NEOX or ORACLE_ROPE_GPTJ.
 * q rows have 576 dims when the lists hold V3.2 records (all of them, and
 * no RoPE table), else 512.
 * Returns 0, or -1 on bad arguments / out of memory. */
int oracle_decode(int32_t H, const uint16_t *q, int64_t q_st, int64_t q_sh,
                  const oracle_cache *caches, const oracle_list *lists, int32_t nlists,
                  const float *sink, const int64_t *positions, const float *cos_sin,
                  int64_t cs_rows, int32_t rope_style, double scale, const int32_t *tokens,
                  int32_t n_tokens, double *out, double *lse, int32_t *kept,
                  uint32_t *checksum, int32_t nthreads) {
  if (H <= 0 || !q || !caches || !lists || nlists < 1 || nlists > 2 || n_tokens < 0) return -1;
  if (rope_style != ORACLE_ROPE_NEOX && rope_style != ORACLE_ROPE_GPTJ) return -1;
  if (cos_sin && !positions) return -1;
  int v32 = 0;
  for (int32_t L = 0; L < nlists; ++L) v32 += caches[L].format == ORACLE_FMT_V32_656;
  if (v32 != 0 && (v32 != nlists || cos_sin)) return -1;
  const int dk = v32 ? ORACLE_DQK_V32 : ORACLE_D;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n_tokens && n_tokens > 0) nthreads = n_tokens;
  oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -1;
  }
  for (int32_t w = 0; w < nthreads; ++w) {
    oracle_job *J = &jobs[w];
    J->H = H; J->q = q; J->q_st = q_st; J->q_sh = q_sh;
    J->caches = caches; J->lists = lists; J->nlists = nlists;
    J->sink = sink; J->positions = positions; J->cos_sin = cos_sin; J->cs_rows = cs_rows;
    J->rope_style = rope_style;
    J->dk = dk;
    J->scale = scale; J->tokens = tokens; J->n_tokens = n_tokens;
    J->out = out; J->lse = lse; J->kept = kept; J->checksum = checksum;
    J->nthreads = nthreads; J->tid = w; J->status = 0;
  }
  /* Positions must index the table. */
  if (cos_sin) {
    for (int32_t i = 0; i < n_tokens; ++i) {
      int64_t p = positions[tokens[i]];
      if (p < 0 || p >= cs_rows) {
        free(jobs);
        free(th);
        return -1;
      }
    }
  }
  int32_t started = 0;
  for (int32_t w = 1; w < nthreads; ++w) {
    if (pthread_create(&th[w], NULL, worker, &jobs[w]) != 0) break;
    started = w;
  }
  worker(&jobs[0]);
  for (int32_t w = 1; w <= started; ++w) pthread_join(th[w], NULL);
  /* Threads that failed to start: run their share here. */
  for (int32_t w = started + 1; w < nthreads; ++w) worker(&jobs[w]);
  int rc = 0;
  for (int32_t w = 0; w < nthreads; ++w)
    if (jobs[w].status) rc = -1;
  free(jobs);
  free(th);
  return rc;
}

/* ------------------------------------------------------------------------
 * V4.1 output epilogue (the swapab page, merge step, after the sink merge:
 * inverse RoPE on dims >= 448, MXFP8 cast with one ue8m0 scale per 32 dims,
 * "o-fused" store).
 */

/* Nearest E4M3 code to y, ties to the code with an even mantissa; |y| past
 * 448 saturates to 448 (the page's cast to fp8 is a saturating one); the
 * sign of y is kept, also for results that round to zero; NaN gives 0x7F.
 * Brute force over the 127 finite magnitudes, whose values increase with the
 * code, so a tie is between codes c and c + 1 and goes to the even one. */
uint8_t oracle_e4m3_encode(double y) {
  if (isnan(y)) return 0x7F;
  const uint8_t sign = signbit(y) ? 0x80 : 0x00;
  const double a = fabs(y);
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c <= 126; ++c) {
    const double d = fabs(oracle_e4m3_value((uint8_t)c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return (uint8_t)(sign | best);
}

/* ue8m0 byte of the smallest power of two >= v (v a positive finite fp32
 * value): with v = f * 2^e, f in [0.5, 1), ceil(log2 v) is e - 1 when
 * f = 0.5 (v a power of two) and e otherwise; biased by 127 and saturated
 * to 0..254 (0xFF is NaN in E8M0). */
uint8_t oracle_ue8m0_ceil(float v) {
  int e = 0;
  const double f = frexp((double)v, &e);
  int E = (f == 0.5) ? e - 1 : e;
  int b = E + 127;
  if (b < 0) b = 0;
  if (b > 254) b = 254;
  return (uint8_t)b;
}

/* out: [n][H][512] fp64 outputs (rows of out from oracle_decode). pos: [n]
 * the rows' positions (read only with cos_sin). cos_sin: fp32 [cs_rows][64]
 * or NULL (no RoPE: no inverse rotation). rope_style: the pairing of the
 * forward rotation. G: heads per output group (divides H).
 *   1. Inverse rotation of dims >= 448 with the row's c = cos[i], s = sin[i]
 *      (the forward rotation with s negated): x1 <- x1 c + x2 s,
 *      x2 <- x2 c - x1 s, pairs as in step 4 of oracle_decode.
 *   2. Each value is rounded to fp32: the page takes the scale and code
 *      decisions in fp32.
 *   3. Per head h and 32-dim chunk cc: amax = max(max_d |x|, 1e-10) and
 *      v = amax * fp32(1/448), a product rounded to fp32; scale byte
 *      E = oracle_ue8m0_ceil(v) (= ceil(log2(amax / 448)) + 127); the code of
 *      x is oracle_e4m3_encode(x * 2^(127 - E)) (the product is exact).
 *   4. o-fused layout: group g = h / G, slot ka = cc * G + h % G;
 *      codes[n][H/G][G*512] at [g][ka*32 + d%32], scales[n][H/G][G*16] at
 *      [g][ka] (one byte per (head, chunk); the page packs them four to an
 *      int32 word, little-endian, which is the same byte order).
 * x_out (optional, [n][H][512] fp32): the values after steps 1-2.
 * Returns 0, or -1 on bad arguments. */
int oracle_mxfp8_epilogue(const double *out, int32_t n, int32_t H, const int64_t *pos,
                          const float *cos_sin, int64_t cs_rows, int32_t rope_style,
                          int32_t G, float *x_out, uint8_t *codes, uint8_t *scales) {
  if (!out || n < 0 || H <= 0 || G <= 0 || H % G != 0 || !codes || !scales) return -1;
  if (cos_sin && !pos) return -1;
  if (rope_style != ORACLE_ROPE_NEOX && rope_style != ORACLE_ROPE_GPTJ) return -1;
  const float inv448 = 1.0f / 448.0f;
  for (int32_t r = 0; r < n; ++r) {
    if (cos_sin && (pos[r] < 0 || pos[r] >= cs_rows)) return -1;
    for (int32_t h = 0; h < H; ++h) {
      double o[ORACLE_D];
      memcpy(o, out + ((int64_t)r * H + h) * ORACLE_D, sizeof(o));
      if (cos_sin) {
        const float *row = cos_sin + pos[r] * 64;
        for (int i = 0; i < ORACLE_ROPE_HALF; ++i) {
          const double c = (double)row[i], sn = (double)row[ORACLE_ROPE_HALF + i];
          int d1, d2;
          if (rope_style == ORACLE_ROPE_GPTJ) {
            d1 = ORACLE_ROPE_START + 2 * i;
            d2 = d1 + 1;
          } else {
            d1 = ORACLE_ROPE_START + i;
            d2 = d1 + ORACLE_ROPE_HALF;
          }
          const double x1 = o[d1], x2 = o[d2];
          o[d1] = x1 * c + x2 * sn;
          o[d2] = x2 * c - x1 * sn;
        }
      }
      float x[ORACLE_D];
      for (int d = 0; d < ORACLE_D; ++d) x[d] = (float)o[d];
      if (x_out) memcpy(x_out + ((int64_t)r * H + h) * ORACLE_D, x, sizeof(x));
      const int32_t g = h / G, hg = h % G;
      for (int cc = 0; cc < ORACLE_D / 32; ++cc) {
        float amax = 0.0f;
        for (int d = 32 * cc; d < 32 * cc + 32; ++d) amax = fmaxf(amax, fabsf(x[d]));
        amax = fmaxf(amax, 1e-10f);
        const float v = amax * inv448;
        const uint8_t E = oracle_ue8m0_ceil(v);
        const int64_t ka = (int64_t)cc * G + hg;
        uint8_t *crow = codes + ((int64_t)r * (H / G) + g) * ((int64_t)G * ORACLE_D);
        for (int d = 32 * cc; d < 32 * cc + 32; ++d)
          crow[ka * 32 + d % 32] = oracle_e4m3_encode(ldexp((double)x[d], 127 - (int)E));
        scales[((int64_t)r * (H / G) + g) * ((int64_t)G * 16) + ka] = E;
      }
    }
  }
  return 0;
}
