// dsa_internal.cuh -- shared definitions of the CUDA library (not part of the
// public ABI): the launch parameter block, the static work schedule, record
// decoding and row selection.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_decode.h"

namespace dsa {

constexpr int kD = 512;          // head dim (K = V row)
constexpr int kTile = 128;       // KV rows per work unit
constexpr int kRopeStart = 448;  // RoPE acts on the last 64 dims
constexpr int kRopeHalf = 32;
constexpr int32_t kPlanMagic = 0x31415344;  // "DSA1"
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum KernelVariant : int32_t { kKernelSimt = 0, kKernelTc = 1 };

// One slot list with the cache it points into.
struct ListArgs {
  const uint8_t *base;   // cache bytes
  int64_t num_slots;     // num_pages * page_size
  int64_t page_stride;   // bytes
  const int32_t *ids;    // [T, idx_stride]
  const int32_t *lens;   // [T]
  int64_t idx_stride;
  int64_t extent;        // bytes of the cache: num_pages * page_stride
  int32_t page_shift;    // log2(page_size)
  int32_t page_mask;     // page_size - 1
  int32_t fmt;           // DSA_REC_*
  int32_t rec;           // record bytes
  int32_t width;
  int32_t tiles;         // ceil(width / kTile)
  int32_t aligned32;     // every record starts on a 32-byte boundary
  int32_t sectors32;     // base and page stride 32-byte aligned (records may not be)
};

struct Params {
  const __nv_bfloat16 *q;
  int64_t q_st, q_sh;          // element strides
  int32_t dqk;                 // key / query dims: 512, or 576 (V3.2 records)
  int32_t pq;                  // plan's producer_q: the producers stage Q (plain form)
  int32_t merge;               // plan's merge_in_run: the run kernel merges split tokens
  int32_t *tok_cnt;            // [HG][T] units of each token done (zeroed per run)
  ListArgs list[2];
  int32_t nlists;
  const float *sink;           // [H] or null
  const int64_t *positions;    // [T] or null
  const float *cos_sin;        // [cs_rows, 64] or null
  int64_t cs_rows;
  float scale;
  float scale_log2;            // scale * log2(e)
  int32_t rope_gptj;           // RoPE pairing: 0 NeoX (448+i, 480+i), 1 GPT-J (448+2i, 449+2i)
  __nv_bfloat16 *out;          // [T, H, 512] (bf16 output), or null with mx_on
  float *lse;                  // [T, H]
  // MXFP8 output (V4.1 epilogue): the decode and combine kernels leave each
  // token's fp32 output in `stage`; the epilogue kernel casts it into the
  // codes and ue8m0 scales of the o-fused layout
  float *stage;                // [T, H, 512] in the workspace, with mx_on
  int32_t mx_on;               // 1: write mx_* instead of out
  int32_t mx_g;                // heads per output group
  uint8_t *mx_data;            // code (t, h, d) at t*mx_st + (h/G)*mx_sg + (c*G + h%G)*32 + d%32, c = d/32
  uint8_t *mx_scale;           // byte (t, h, c) at 4*(t*mx_sst + (h/G)*mx_ssg + (ka/4)*mx_ssw) + ka%4, ka = c*G + h%G
  int64_t mx_st, mx_sg;        // bytes
  int64_t mx_sst, mx_ssg, mx_ssw;   // int32 words
  // schedule (copied from the plan)
  int32_t T, H, hpg, HG, tpt, upc, C;
  int64_t U;
  // workspace
  int64_t *bounds;             // [C+1]: CTA c owns units [bounds[c], bounds[c+1])
  int32_t balance;             // 1: live-tile balanced ranges, 0: c*upc
  long long wait_budget;       // SM cycles per bounded device wait (0: the kernel's default)
  int32_t *status;             // device status word
  int32_t *sel;                // [T][2]: kept rows, checksum
  float *part_lse;             // [HG][2C][hpg]
  int32_t *part_sel;           // [2C][2]
  float *part_o;               // [HG][2C][hpg][512]
};

// ---------------------------------------------------------------- schedule
// Units are (token, tile) pairs in token-major order. A tile is live when its
// first row lies below min(len, width) of its list; dead tiles cost nothing
// but a skip. The C CTAs of a head group split the units into contiguous
// ranges. With p.balance the ranges hold equal work (FlashMLA's
// decoding-schedule idea, sparse_decode.h get_decoding_sched_meta): with
// kCostTile per live tile and kCostToken per token that has any (its Q
// staging and finalize), total L, CTA c starts at the unit where cost
// floor(c L / C) falls (CTA 0 at unit 0); when L / (kCostTile + kCostToken)
// < C, or without p.balance, CTA c owns [c*upc, (c+1)*upc) clipped to U.
// Inside a CTA, the
// first and last tokens may be partial ("split"); their partial results go
// to slot 2c (the first token) and 2c+1 (the last token, when different).
struct Segment {
  int32_t t;        // token
  int64_t u_begin;  // first unit
  int64_t u_end;    // one past the last unit
  bool whole;       // covers every unit of the token
  int32_t slot;     // partial slot when !whole
};

// live tiles of list L for token t
__device__ inline int32_t live_tiles(const ListArgs &L, int64_t t) {
  int32_t n = __ldg(L.lens + t);
  n = n < 0 ? 0 : (n > L.width ? L.width : n);
  return (n + kTile - 1) / kTile;
}
__device__ inline int64_t live_tiles_token(const Params &p, int64_t t) {
  return live_tiles(p.list[0], t) + (p.nlists > 1 ? live_tiles(p.list[1], t) : 0);
}
// Work of a token in cost units: kCostTile per live tile plus kCostToken
// for the per-token steps (Q staging, finalize) when it has any live tile.
constexpr int64_t kCostTile = 4, kCostToken = 10;
__device__ inline int64_t token_cost(int64_t live) {
  return live > 0 ? kCostTile * live + kCostToken : 0;
}

// Unit range [u0, u1) of CTA c. Called by every thread of the block (it
// synchronizes the block; blockDim.x a multiple of 32, at most 1024); scr:
// shared scratch of blockDim.x + 2 + blockDim.x / 32 int64. Also publishes
// the range to p.bounds (both ends, so that a CTA merging a split token
// finds every part's range written by that part) for the merge.
__device__ inline void cta_range(const Params &p, int32_t c, int64_t *scr, int64_t &u0,
                                 int64_t &u1) {
  const int n = blockDim.x, tid = threadIdx.x;
  if (!p.balance) {   // even split of the units
    u0 = (int64_t)c * p.upc;
    u0 = u0 < p.U ? u0 : p.U;
    u1 = u0 + p.upc < p.U ? u0 + p.upc : p.U;
    if (tid == 0) {
      p.bounds[c] = u0;
      p.bounds[c + 1] = u1;   // also written by CTA c + 1 (same value)
    }
    return;
  }
  const int64_t T = p.T;
  const int64_t t0 = T * tid / n, t1 = T * (tid + 1) / n;
  int64_t sum = 0;
  for (int64_t t = t0; t < t1; ++t) sum += token_cost(live_tiles_token(p, t));
  // inclusive scan over the threads' token chunks: within each warp by
  // shuffles, then over the warp totals (one warp), then their offsets
  const int lane = tid & 31, wid = tid >> 5, nw = n >> 5;
  int64_t v = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += y;
  }
  int64_t *wsum = scr + n + 2;   // [nw] warp totals, then their inclusive prefixes
  if (lane == 31) wsum[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int64_t w = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < nw) wsum[lane] = w;
  }
  __syncthreads();
  scr[tid] = v + (wid > 0 ? wsum[wid - 1] : 0);
  __syncthreads();
  const int64_t L = scr[n - 1];   // total cost
  if (tid < 2) {
    const int64_t cc = (int64_t)c + tid;
    // boundaries at least kCostToken + kCostTile cost units apart fall on
    // distinct units, so no CTA below ce is left empty
    const int64_t cmax = L / (kCostToken + kCostTile);
    const int64_t ce = cmax < 1 ? 1 : (cmax < p.C ? cmax : p.C);
    int64_t b;
    if (ce < p.C) {
      // too little work to keep every CTA busy at that spacing: the even
      // split keeps all C CTAs (every CTA has units; live or not)
      b = cc * p.upc < p.U ? cc * p.upc : p.U;
    } else if (cc == 0) {
      b = 0;
    } else if (cc >= ce) {
      b = p.U;
    } else {
      const int64_t li = cc * L / ce;   // cost unit that starts CTA cc
      int lo = 0, hi = n - 1;           // first chunk whose inclusive prefix exceeds li
      while (lo < hi) {
        const int mid = (lo + hi) / 2;
        if (scr[mid] > li) hi = mid; else lo = mid + 1;
      }
      int64_t acc = lo > 0 ? scr[lo - 1] : 0;
      b = p.U;
      for (int64_t t = T * lo / n, te = T * (lo + 1) / n; t < te; ++t) {
        const int64_t n0 = live_tiles(p.list[0], t);
        const int64_t lt = n0 + (p.nlists > 1 ? live_tiles(p.list[1], t) : 0);
        const int64_t ct = token_cost(lt);
        if (li < acc + ct) {   // the token's fixed cost maps to its first live tile
          int64_t k = (li - acc - kCostToken) / kCostTile;
          k = k < 0 ? 0 : k;
          b = t * p.tpt + (k < n0 ? k : p.list[0].tiles + (k - n0));
          break;
        }
        acc += ct;
      }
    }
    scr[n + tid] = b;
  }
  __syncthreads();
  u0 = scr[n];
  u1 = scr[n + 1];
  __syncthreads();   // scratch free again
  if (tid == 0) {
    p.bounds[c] = u0;
    p.bounds[c + 1] = u1;   // also written by CTA c + 1 (same value)
  }
}

__device__ inline Segment make_segment(const Params &p, int32_t c, int32_t t, int64_t u0,
                                       int64_t u1) {
  int64_t ts = (int64_t)t * p.tpt, te = ts + p.tpt;
  Segment s;
  s.t = t;
  s.u_begin = u0 > ts ? u0 : ts;
  s.u_end = u1 < te ? u1 : te;
  s.whole = (s.u_begin == ts) && (s.u_end == te);
  int32_t tf = (int32_t)(u0 / p.tpt);
  s.slot = 2 * c + (t == tf ? 0 : 1);
  return s;
}

// Unit -> (list, first row).
__device__ inline void unit_tile(const Params &p, int64_t u, int32_t &lid, int32_t &row0) {
  int32_t k = (int32_t)(u % p.tpt);
  if (k < p.list[0].tiles) {
    lid = 0;
    row0 = k * kTile;
  } else {
    lid = 1;
    row0 = (k - p.list[0].tiles) * kTile;
  }
}

// ---------------------------------------------------------------- selection
// A list position r of token t names a row iff r < clamp(len, 0, width) and
// 0 <= id < num_slots (vLLM swapab page, SwapABDecodeKernel.stage_inputs).
__device__ inline int32_t list_limit(const ListArgs &L, int32_t t) {
  int32_t len = __ldg(L.lens + t);
  len = len < 0 ? 0 : len;
  return len < L.width ? len : L.width;
}

__device__ inline bool slot_valid(const ListArgs &L, int32_t r, int32_t limit, int32_t sid) {
  return r < limit && sid >= 0 && (int64_t)sid < L.num_slots;
}

// Record address: page = sid >> page_shift, offset = sid & page_mask.
__device__ inline const uint8_t *record_ptr(const ListArgs &L, int32_t sid) {
  int64_t blk = (int64_t)(sid >> L.page_shift);
  int64_t off = (int64_t)(sid & L.page_mask);
  return L.base + blk * L.page_stride + off * L.rec;
}

// MurmurHash3 32-bit finalizer; feeds the row-selection checksum.
__device__ inline uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}
__device__ inline uint32_t row_hash(int32_t sid, int32_t r, int32_t lid) {
  return fmix32((uint32_t)sid * 0x9E3779B1u + 2u * (uint32_t)r + (uint32_t)lid);
}

// ---------------------------------------------------------------- decoding
// e4m3 (bias 7, subnormal below exponent field 1) -> fp32, exact: place the
// 7 magnitude bits at the top of the fp32 exponent/mantissa fields, which
// reads as 2^(e-127) * (1 + m/8) (or the fp32 subnormal m * 2^-129 when e is
// 0), then multiply by 2^120. Needs denormals kept (no -ftz).
__device__ inline float e4m3_to_f32(uint32_t code) {
  float mag = __uint_as_float((code & 0x7Fu) << 20) * 1.329227995784916e36f;  // 2^120
  return (code & 0x80u) ? -mag : mag;
}

// ue8m0 scale byte b -> 2^(b - 127) as fp32, exact (b = 0 is the fp32
// subnormal 2^-127); b = 0xFF is NaN.
__device__ inline float ue8m0_to_f32(uint32_t b) {
  b &= 0xFFu;
  if (b == 0xFFu) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(b ? (b << 23) : 0x00400000u);
}

// e2m1 (bias 1, subnormal at exponent field 0) -> fp32, exact, same trick
// with 2^126.
__device__ inline float e2m1_to_f32(uint32_t nib) {
  float mag = __uint_as_float((nib & 0x7u) << 22) * 8.507059173023462e37f;  // 2^126
  return (nib & 0x8u) ? -mag : mag;
}

// One-time per-device kernel set-up (function attributes): `f` runs on the
// first launch of kernel variant `bit` on the current device, later launches
// skip it (they may be captured into a CUDA graph, where no set-up call is
// wanted). Thread-safe. Bits in use: tensor-core kernels 0-2 (plain), 20-22
// (V4.1 options), 24-26 (exact-budget waits), 28-30 and 32-34 (MODEL1 records),
// 36-37 (V3.2 records), 40-42 (head groups sharing tiles), 46 and 50
// (producers staging Q, with and without shared tiles), SIMT kernels 8-11,
// combine 16-18.
cudaError_t dsa_configure_once(int bit, cudaError_t (*f)(void *), void *arg);

// Programmatic dependent launch: the decode kernels let the combine grid be
// scheduled early; the combine kernel waits for their completion (and
// memory) before reading the partials.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ inline float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// ---------------------------------------------------------------- MXFP8 out
// The V4.1 output epilogue (the swapab page's merge step): inverse GPT-J
// RoPE on dims >= 448, then per head and 32-dim chunk an ue8m0 scale
// E = ceil(log2(max(amax, 1e-10) * fp32(1/448))) + 127 and e4m3 codes of
// x * 2^(127 - E), stored in the o-fused layout.

// ue8m0 byte of the smallest power of two >= v, v a positive normal fp32
// value: the biased exponent field, plus one unless the mantissa field is
// zero (then v is that power of two); saturated at 254 (0xFF is NaN).
__device__ __forceinline__ uint32_t ue8m0_ceil(float v) {
  const uint32_t b = __float_as_uint(v);
  const uint32_t e = ((b >> 23) & 0xFFu) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
  return e > 254u ? 254u : e;
}
// 2^(127 - E) for a scale byte E in [1, 254] (fp32 bits (254 - E) << 23).
__device__ __forceinline__ float ue8m0_inverse(uint32_t E) { return __uint_as_float((254u - E) << 23); }

// Two fp32 values -> e4m3 codes (round to nearest even, saturating to
// +-448): lo in bits 0..7, hi in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// o-fused addresses of head h (absolute), 32-dim chunk c of token t.
__device__ __forceinline__ uint8_t *mx_chunk(const Params &p, int64_t t, int h, int c) {
  const int g = h / p.mx_g, ka = c * p.mx_g + (h - g * p.mx_g);
  return p.mx_data + t * p.mx_st + (int64_t)g * p.mx_sg + (int64_t)ka * 32;
}
__device__ __forceinline__ uint8_t *mx_scale_byte(const Params &p, int64_t t, int h, int c) {
  const int g = h / p.mx_g, ka = c * p.mx_g + (h - g * p.mx_g);
  return p.mx_scale + 4 * (t * p.mx_sst + (int64_t)g * p.mx_ssg + (int64_t)(ka >> 2) * p.mx_ssw) +
         (ka & 3);
}

// Table row of token t for the inverse rotation (null without RoPE or for
// NeoX, whose inverse the MXFP8 path does not take); a position outside the
// table uses row 0, as the Q staging does.
__device__ __forceinline__ const float *mx_rope_row(const Params &p, int64_t t) {
  if (!p.cos_sin || !p.rope_gptj) return nullptr;
  int64_t pos = __ldg(p.positions + t);
  if (pos < 0 || pos >= p.cs_rows) pos = 0;
  return p.cos_sin + pos * 64;
}

// Status word: first failure wins.
__device__ inline void report_status(int32_t *status, int32_t code) {
  atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- checking build
// Built with -DDSA_DEBUG (libdsa_decode_debug.so), the kernels check every
// record, slot-id, Q and table read, every output store and every store into
// a shared-memory tile against the extent it must stay in. A failed check
// skips the access (a record read becomes a row that is not kept) and
// records DSA_ERR_BOUNDS in the status word and the check's kind in word 1 of
// the status block (first failure wins). The release build compiles none of
// it (kDebug is false, every check folds to true).
enum DebugKind : int32_t {
  kDbgRecord = 1, kDbgIds = 2, kDbgQ = 3, kDbgTable = 4, kDbgOut = 5, kDbgPartial = 6,
  kDbgSmemKv = 7, kDbgSmemQ = 8, kDbgSmemP = 9, kDbgSel = 10
};
#ifdef DSA_DEBUG
constexpr bool kDebug = true;
#else
constexpr bool kDebug = false;
#endif
__device__ __forceinline__ bool dbg_ok(int32_t *status, bool ok, int32_t kind) {
  if (!kDebug || ok) return true;
  if (atomicCAS(status, 0, DSA_ERR_BOUNDS) == 0) atomicExch(status + 1, kind);
  return false;
}

}  // namespace dsa

// Launchers (defined in the kernel translation units).
cudaError_t dsa_launch_simt(const dsa::Params &p, cudaStream_t stream);
cudaError_t dsa_launch_tc(const dsa::Params &p, cudaStream_t stream);
bool dsa_tc_supports(int heads_per_group);
cudaError_t dsa_launch_combine(const dsa::Params &p, cudaStream_t stream);
cudaError_t dsa_launch_mx_epilogue(const dsa::Params &p, cudaStream_t stream);
