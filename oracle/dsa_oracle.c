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
 *      bytes then 4 little-endian fp32 scales, one per 128 dims; the NVFP4
 *      record holds 256 bytes of e2m1 nibbles then 32 e4m3 scales, one per 16
 *      dims, element 2i in the low nibble of byte i and 2i+1 in the high one).
 *      k[d] = code(d) * scale(d).
 *   4. Q.  q = bf16 value of q[t, h, :] in fp64. With RoPE on, the last 64
 *      dims are rotated NeoX style (first half against second half) by the
 *      fp32 table row cos_sin[positions[t]] = [cos(32) | sin(32)]:
 *      x1 = q[448+i], x2 = q[480+i]; q[448+i] = x1 c - x2 s,
 *      q[480+i] = x2 c + x1 s.
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

#define ORACLE_D 512
#define ORACLE_ROPE_START 448
#define ORACLE_ROPE_HALF 32

enum { ORACLE_FMT_FP8_528 = 0, ORACLE_FMT_NVFP4_288 = 1 };

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
  return format == ORACLE_FMT_FP8_528 ? 528 : 288;
}

/* Step 3: one record -> 512 fp64 values. */
void oracle_dequant_record(const uint8_t *rec, int32_t format, double *k) {
  if (format == ORACLE_FMT_FP8_528) {
    for (int d = 0; d < ORACLE_D; ++d)
      k[d] = oracle_e4m3_value(rec[d]) * le_f32(rec + 512 + 4 * (d / 128));
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
                           int32_t t, double *K, int64_t n, uint32_t *sum) {
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
    oracle_dequant_record(rec, c->format, K + n * ORACLE_D);
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
    n = gather_list(&J->caches[L], &J->lists[L], L, t, K, n, &sum);
  J->kept[i] = (int32_t)n;
  J->checksum[i] = sum;

  double q[ORACLE_D];
  for (int32_t h = 0; h < J->H; ++h) {
    const uint16_t *qh = J->q + (int64_t)t * J->q_st + (int64_t)h * J->q_sh;
    for (int d = 0; d < ORACLE_D; ++d) q[d] = bf16_value(qh[d]);
    if (J->cos_sin) {
      int64_t pos = J->positions[t];
      const float *row = J->cos_sin + pos * 64;
      for (int i2 = 0; i2 < ORACLE_ROPE_HALF; ++i2) {
        double c = (double)row[i2], sn = (double)row[ORACLE_ROPE_HALF + i2];
        double x1 = q[ORACLE_ROPE_START + i2];
        double x2 = q[ORACLE_ROPE_START + ORACLE_ROPE_HALF + i2];
        q[ORACLE_ROPE_START + i2] = x1 * c - x2 * sn;
        q[ORACLE_ROPE_START + ORACLE_ROPE_HALF + i2] = x2 * c + x1 * sn;
      }
    }
    /* Step 5: scores. */
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      const double *k = K + j * ORACLE_D;
      double dot = 0.0;
      for (int d = 0; d < ORACLE_D; ++d) dot += q[d] * k[d];
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
      const double *k = K + j * ORACLE_D;
      for (int d = 0; d < ORACLE_D; ++d) o[d] += w * k[d];
    }
  }
}

static void *worker(void *arg) {
  oracle_job *J = (oracle_job *)arg;
  int64_t maxrows = 0;
  for (int32_t L = 0; L < J->nlists; ++L) maxrows += J->lists[L].width;
  double *K = (double *)malloc((size_t)(maxrows > 0 ? maxrows : 1) * ORACLE_D * sizeof(double));
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
 * checksum[n_tokens]. Returns 0, or -1 on bad arguments / out of memory. */
int oracle_decode(int32_t H, const uint16_t *q, int64_t q_st, int64_t q_sh,
                  const oracle_cache *caches, const oracle_list *lists, int32_t nlists,
                  const float *sink, const int64_t *positions, const float *cos_sin,
                  int64_t cs_rows, double scale, const int32_t *tokens, int32_t n_tokens,
                  double *out, double *lse, int32_t *kept, uint32_t *checksum,
                  int32_t nthreads) {
  if (H <= 0 || !q || !caches || !lists || nlists < 1 || nlists > 2 || n_tokens < 0) return -1;
  if (cos_sin && !positions) return -1;
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
