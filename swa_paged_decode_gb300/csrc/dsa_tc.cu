// dsa_tc.cu -- fused gather + dequant + attention on sm_103a tensor cores.
//
// One persistent CTA per SM walks a contiguous range of (token, 128-row tile)
// units with three warp-specialised roles joined by mbarriers:
//
//   producers (warps 8-15)  gather: the tile's 128 records, one tile ahead,
//            held in registers (the two halves of a row in adjacent lanes;
//            32-byte loads where a record starts on a 32-byte boundary, the
//            aligned 32-byte sectors around fp8 records 16 bytes off that
//            grid, predicated 16-byte loads otherwise); dequant: records ->
//            f16 K-major tile in shared memory, 128-byte swizzle (16-byte
//            chunk c of row r at chunk c ^ (r % 8)), written one 128-dim block
//            at a time as soon as the PV MMAs of the previous tile release
//            it. NVFP4: e2m1 * e4m3 scale (exact in f16). fp8: e4m3 * the
//            fp32 block scale rounded to f16, the product rounded to f16
//            (relative error <= 2^-11 per element). fp8 with ue8m0 scales
//            (the V4.1 record): e4m3 * 2^(b - 127), exact in f16 for scale
//            exponents in [-15, 7].
//   MMA issue (one thread of warp 0)  swap-AB tcgen05.mma kind::f16:
//            S[128 rows, H] = K[128, 512] . Q[H, 512]^T into TMEM, issued back
//            to back once the tile has landed; then O^T[512, H] += K^T . P in four
//            128-dim M blocks, A read MN-major from the same tile. Commits
//            release tile blocks (to the producers) and S / O (to softmax).
//   softmax (warps 0-7)     one TMEM lane (= one KV row) and half of the heads
//            per thread; scores x = S * scale * log2e;
//            base-2 running max per head that moves only when a score passes
//            it by 2^8 (then O in TMEM and the partial sums are rescaled);
//            P = 2^(x - m) as f16. Also stages Q (NeoX or GPT-J RoPE,
//            per-head power-of-two prescale into f16) and, per token,
//            reduces the sums, folds the sink into the denominator and writes
//            out (bf16) and lse (fp32) -- or, for MXFP8 output, the fp32
//            output to a staging area that a separate kernel casts -- or an
//            fp32 partial for a token split over CTAs, merged later by the
//            combine kernel.
//
// The V4.1 options (ue8m0 records, GPT-J RoPE, MXFP8 staging) exist only in
// the kExt instantiation; the plain one compiles without them.
//
// Tiles whose first row lies past min(len, width) are skipped by every role
// (each evaluates the same predicate from the lengths), so all roles walk the
// same sequence of tiles and tokens. Every mbarrier wait is bounded; when one
// gives up the CTA records DSA_ERR_TIMEOUT, later waits return at once and no
// further MMA is issued, while every role still walks its loops to the end
// (named barriers keep matching).
//
// Design sources (prior art, re-derived for this GPU): the vLLM
// "swapab_decode_attn" page (SwapABDecodeKernel: swap-AB tcgen05 tiles of 128
// KV rows, K-major SW128 KV tile read MN-major for PV, predicated 16-byte
// record loads, base-2 softmax), FlashMLA's sparse_decode.h page (split-KV
// partials + combine).
#include "dsa_internal.cuh"
#include "tc_ptx.cuh"

namespace dsa {

constexpr int kSmWarps = 8;                    // softmax / epilogue / MMA issue
constexpr int kPrWarps = 8;                    // producers
constexpr int kTcThreads = 32 * (kSmWarps + kPrWarps);
// Register split (per thread): the kernel is launched with 128; softmax
// warpgroups raise theirs and producer warpgroups drop theirs by the same
// amount, so the split sums to exactly the launch allocation. 64 heads per
// group: 152 / 104 (the softmax side needs the room); 16 and 32: 144 / 112,
// where ptxas reports no spills.
constexpr int kLaunchRegs = 128;
constexpr long long kWaitBudget = 4000000000ll;  // SM cycles (~2 s) per wait
constexpr float kRescaleSlack = 8.0f;            // log2 headroom of the running max
// Row exponents: an fp8 row is written to the f16 tile as k * 2^-e, e the
// exponent of its largest block scale (so its largest scale lies in [1, 2)),
// clamped to [-kRowExpMax, kRowExpMax]; the softmax puts 2^e back exactly.
constexpr int kRowExpMax = 48;
constexpr int32_t kRowInvalid = INT32_MIN;       // row record of a row that is not kept
constexpr float kMaxInit = -1e30f;               // running max before any kept row

template <int HPG, bool V32 = false>
struct TcCfg {
  static constexpr int kSmRegs = HPG == 64 ? 152 : 144;
  static constexpr int kPrRegs = 2 * kLaunchRegs - kSmRegs;
  static constexpr int kHalf = HPG / 2;                  // heads per softmax thread
  static constexpr int kPRow = HPG * 2;                  // bytes per P row
  static constexpr uint32_t kPBytes = 128 * kPRow;
  static constexpr int kQD = V32 ? 576 : 512;            // Q (and key) dims
  static constexpr uint32_t kKV = 0;                     // 128 x 512 f16 = 128 KiB
  static constexpr uint32_t kKR = 131072;                // V32: [128 x 64] f16, key dims 512..575
  static constexpr uint32_t kQ = kKR + (V32 ? 16384 : 0);   // HPG x kQD f16 (k-blocks of 64 dims)
  static constexpr uint32_t kP = kQ + HPG * kQD * 2;     // [128 x HPG] f16
  static constexpr uint32_t kRho = kP + kPBytes;         // [128] int32 row exponent, kRowInvalid: not kept
  static constexpr uint32_t kHeadF = kRho + 1024;        // [64] f32 per-head score factor
  static constexpr uint32_t kM = kHeadF + 256;           // [64] running max (log2)
  static constexpr uint32_t kRed = kM + 256;             // [4][64] f32
  static constexpr uint32_t kMisc = kRed + 1024;         // mbarriers, counters, tmem base
  static constexpr uint32_t kBytes = kMisc + 256;   // bars 72 B, abort, tmem, counters
  static constexpr uint32_t kSmem = kBytes + 1024 > 232448u ? 232448u : kBytes + 1024;
  static constexpr uint32_t kCols = HPG == 16 ? 128 : (HPG == 32 ? 256 : 512);
  static constexpr uint32_t kColS = 0;                   // S block b at b*HPG
  static constexpr uint32_t kColO = 4 * HPG;             // O block mb at (4+mb)*HPG
  static constexpr uint32_t kPSwz = HPG == 64 ? tc::kSwz128 : (HPG == 32 ? tc::kSwz64 : tc::kSwz32);
  static constexpr uint32_t kIdQK = tc::idesc_f16(128, HPG, false, false);
  static constexpr uint32_t kIdPV = tc::idesc_f16(128, HPG, true, true);
  static_assert(kBytes <= 232448u, "shared memory layout exceeds 227 KiB");
};

// mbarrier slots in the misc area
enum Bar : int {
  kBarKvFull = 0,   // producers -> MMA / softmax: the whole tile written
  kBarKvFree = 1,   // [4] MMA commit -> producers: 128-dim block no longer read
  kBarSFull = 5,    // MMA commit -> softmax: S ready (and every earlier MMA done)
  kBarOFinal = 6,   // MMA commit -> softmax: last PV of a token done
  kBarDrain = 7,    // MMA commit -> issuer: every MMA issued so far done (abort path)
  kBarDrainQK = 8,  // producers' QK commits -> themselves: their MMAs done (abort path)
  kNumBars = 9
};
constexpr uint32_t kMiscAbort = 8 * kNumBars;        // int32
constexpr uint32_t kMiscTmem = kMiscAbort + 4;       // uint32
constexpr uint32_t kMiscCnt = kMiscAbort + 8;        // [4][2] uint32: kept rows / checksum
constexpr uint32_t kMiscQk = kMiscCnt + 32;          // uint32: producer warps done with opening tiles
// Kept-row records ride in 4 slots indexed by the ordinal of the token among
// the tokens with work: producers can be at most two such tokens ahead of the
// softmax warps that read (and clear) a slot.

__device__ __forceinline__ uint32_t sw128_off(int r, int kb, int ci, uint32_t kb_bytes) {
  return (uint32_t)kb * kb_bytes + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
         (uint32_t)((ci ^ (r & 7)) << 4);
}

template <int HPG>
__device__ __forceinline__ uint32_t p_off(int r, int ci) {
  if constexpr (HPG == 64)
    return (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u + (uint32_t)((ci ^ (r & 7)) << 4);
  else if constexpr (HPG == 32)
    return (uint32_t)(r >> 3) * 512u + (uint32_t)(r & 7) * 64u +
           (uint32_t)((ci ^ ((r & 7) >> 1)) << 4);
  else
    return (uint32_t)(r >> 3) * 256u + (uint32_t)(r & 7) * 32u +
           (uint32_t)((ci ^ ((r & 7) >> 2)) << 4);
}

// Position in the CTA's unit range, stepped without 64-bit divisions; keeps
// min(len, width) of both lists for the current token.
struct Cursor {
  int64_t u;
  int32_t t, k;        // token, tile index within the token
  int32_t lim0, lim1;  // row limits of the two lists for token t
};
__device__ __forceinline__ void cursor_limits(const Params &p, Cursor &c) {
  if (c.t < p.T) {
    c.lim0 = list_limit(p.list[0], c.t);
    c.lim1 = p.nlists > 1 ? list_limit(p.list[1], c.t) : 0;
  } else {
    c.lim0 = c.lim1 = 0;
  }
}
__device__ __forceinline__ Cursor cursor_at(const Params &p, int64_t u) {
  Cursor c;
  c.u = u;
  c.t = (int32_t)(u / p.tpt);
  c.k = (int32_t)(u - (int64_t)c.t * p.tpt);
  cursor_limits(p, c);
  return c;
}
__device__ __forceinline__ void cursor_step(const Params &p, Cursor &c) {
  ++c.u;
  if (++c.k == p.tpt) {
    c.k = 0;
    ++c.t;
    cursor_limits(p, c);
  }
}
__device__ __forceinline__ void cursor_tile(const Params &p, const Cursor &c, int32_t &lid,
                                            int32_t &row0) {
  if (c.k < p.list[0].tiles) {
    lid = 0;
    row0 = c.k * kTile;
  } else {
    lid = 1;
    row0 = (c.k - p.list[0].tiles) * kTile;
  }
}
// A tile is worked on iff its first row lies below min(len, width).
__device__ __forceinline__ bool cursor_live(const Params &p, const Cursor &c) {
  int32_t lid, row0;
  cursor_tile(p, c, lid, row0);
  return row0 < (lid == 0 ? c.lim0 : c.lim1);
}
// Advance to the next live unit below u1 (or to u1).
__device__ __forceinline__ void cursor_next_live(const Params &p, Cursor &c, int64_t u1) {
  do {
    cursor_step(p, c);
  } while (c.u < u1 && !cursor_live(p, c));
}
__device__ __forceinline__ void cursor_first_live(const Params &p, Cursor &c, int64_t u1) {
  if (c.u < u1 && !cursor_live(p, c)) cursor_next_live(p, c, u1);
}

// fp32 block scale -> f16x2 (both halves = the scale rounded to f16).
__device__ __forceinline__ uint32_t scale_f16x2(float s) {
  const uint32_t hb = (uint32_t)__half_as_ushort(__float2half_rn(s));
  return hb | (hb << 16);
}

// 2^e as fp32 for an integer e in [-126, 127] (exact).
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// Row exponent from the largest biased exponent field (8 bits, bias 127) of
// a row's block scales: e = field - 127, clamped to [-kRowExpMax, kRowExpMax].
__device__ __forceinline__ int row_exp(uint32_t field) {
  const int e = (int)field - 127;
  return e < -kRowExpMax ? -kRowExpMax : (e > kRowExpMax ? kRowExpMax : e);
}

// ---------------------------------------------------------------- producer
// Thread (producer warp pw, lane l): row 32*(pw%4) + l, half j = pw/4 of the
// record's 16-byte chunks: c = 4m + 2j + e (e in {0,1}) -- whole sectors.
// One row half of a tile held in registers. Pair layout (pl): d[2m], d[2m+1]
// are the thread's 16-byte chunks 4m+2j and 4m+2j+1. fp8: m = 0..7, the 4
// fp32 scales in d[17]; NVFP4: m = 0..3, the 32 e4m3 scales in d[8], d[9].
// Sector layout (fp8 records 16 bytes off the 32-byte grid, !pl): d[2k],
// d[2k+1] = 32-byte sector 2k + j of the grid that starts 16 bytes before
// the record (sector s holds chunks 2s-1 and 2s); lane j = 0 also holds
// sector 16 (chunk 31 and the scales) in d[16], d[17]. The two lanes of a
// row rebuild their pairs with one shuffle per pair (dequant_block).
// MODEL1 records (kM1): d[i] = chunk A[2i + j], i = 0..17, of the 16-byte
// grid that starts at the record (pl: the record is 16-byte aligned) or 8
// bytes before it (odd slots of a 16-byte aligned page); record chunk c
// (bytes 16c .. 16c+16) is A[c], or off the grid the upper half of A[c] and
// the lower half of A[c+1], which the row's other lane holds. tail = record
// bytes 568..583: the last two bf16 words, the 7 scale bytes, the unused one.
struct Gather {
  uint4 d[18];
  uint4 tail;
  uint4 rp[4];   // V3.2 records: this lane's 32 bf16 key dims 512 + 32j ..
  int32_t sid;
  int32_t r;
  bool ok;
  bool pl;
};

template <bool kM1, bool kV32>
__device__ __forceinline__ void issue_loads(const Params &p, const Cursor &c, int32_t sid, int row,
                                            int j, Gather &g) {
  int32_t lid, row0;
  cursor_tile(p, c, lid, row0);
  const ListArgs &L = p.list[lid];
  g.r = row0 + row;
  g.sid = sid;
  g.ok = slot_valid(L, g.r, lid == 0 ? c.lim0 : c.lim1, sid);
  if (kDebug && g.ok) {   // checking build: every byte the loads below touch
    const uint8_t *rec = record_ptr(L, sid);
    const uintptr_t ra = reinterpret_cast<uintptr_t>(rec);
    int back = 0;   // bytes read before the record (realigned layouts)
    if (kM1 && L.fmt == DSA_REC_MODEL1_584)
      back = (ra & 15u) ? 8 : 0;
    else if (L.fmt != DSA_REC_NVFP4_288 && (ra & 31u) != 0 && L.sectors32)
      back = 16;
    g.ok = dbg_ok(p.status, rec - back >= L.base && rec + L.rec <= L.base + L.extent, kDbgRecord);
  }
  const uint4 z = make_uint4(0, 0, 0, 0);
  g.pl = true;
  if (kM1 && L.fmt == DSA_REC_MODEL1_584) {   // 584-byte records, 8-byte aligned
    if (g.ok) {
      const uint8_t *rec = record_ptr(L, sid);
      g.pl = (reinterpret_cast<uintptr_t>(rec) & 15u) == 0;
      // off the grid the record is an odd slot, so the 8 bytes before it
      // belong to the previous slot of the same page
      const uint8_t *a = g.pl ? rec : rec - 8;
#pragma unroll
      for (int i = 0; i < 18; ++i) g.d[i] = tc::ldg_nc_v4(a + 16 * (2 * i + j));
      const uint2 t0 = tc::ldg_nc_v2(rec + 568), t1 = tc::ldg_nc_v2(rec + 576);
      g.tail = make_uint4(t0.x, t0.y, t1.x, t1.y);
    } else {
#pragma unroll
      for (int k = 0; k < 18; ++k) g.d[k] = z;
      g.tail = z;
    }
    return;
  }
  if (L.fmt != DSA_REC_NVFP4_288) {   // both 528-byte fp8 records (and V3.2's first 528 bytes)
    if constexpr (kV32) {   // bytes 528..655: lane j takes 64 of them (16-byte aligned)
      const uint8_t *rec = record_ptr(L, sid);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        g.rp[i] = g.ok ? tc::ldg_nc_v4(rec + 528 + 64 * j + 16 * i) : make_uint4(0, 0, 0, 0);
    }
    if (g.ok) {
      const uint8_t *rec = record_ptr(L, sid);
      if ((reinterpret_cast<uintptr_t>(rec) & 31u) == 0) {   // chunk pairs are whole 32-byte sectors
#pragma unroll
        for (int m = 0; m < 8; ++m) tc::ldg_nc_v8(rec + 64 * m + 32 * j, g.d[2 * m], g.d[2 * m + 1]);
        g.d[17] = tc::ldg_nc_v4(rec + 512);
      } else if (L.sectors32) {
        // 16 bytes off the grid (an odd slot of a 32-byte aligned page, so
        // the sector that starts 16 bytes before the record lies in the page)
        g.pl = false;
        const uint8_t *base = rec - 16;
#pragma unroll
        for (int k = 0; k < 8; ++k) tc::ldg_nc_v8(base + 32 * (2 * k + j), g.d[2 * k], g.d[2 * k + 1]);
        if (j == 0) tc::ldg_nc_v8(base + 32 * 16, g.d[16], g.d[17]);
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k)
          g.d[k] = tc::ldg_nc_v4(rec + 16 * (4 * (k >> 1) + 2 * j + (k & 1)));
        g.d[17] = tc::ldg_nc_v4(rec + 512);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 18; ++k) g.d[k] = z;
    }
  } else {
    if (g.ok && L.aligned32) {   // whole 32-byte sectors per request
      const uint8_t *rec = record_ptr(L, sid);
#pragma unroll
      for (int m = 0; m < 4; ++m) tc::ldg_nc_v8(rec + 64 * m + 32 * j, g.d[2 * m], g.d[2 * m + 1]);
      tc::ldg_nc_v8(rec + 256, g.d[8], g.d[9]);
    } else if (g.ok) {
      const uint8_t *rec = record_ptr(L, sid);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        g.d[k] = tc::ldg_nc_v4(rec + 16 * (4 * (k >> 1) + 2 * j + (k & 1)));
      g.d[8] = tc::ldg_nc_v4(rec + 256);
      g.d[9] = tc::ldg_nc_v4(rec + 272);
    } else {
#pragma unroll
      for (int k = 0; k < 10; ++k) g.d[k] = z;
    }
  }
}

// V3.2 records: this lane's 32 bf16 key dims 512 + 32j .. (g.rp) times the
// row's 2^-e into the [128 x 64] f16 tile of dims 512..575 (K-major, one
// SW128 k-block; chunks 4j .. 4j + 3 of the row).
__device__ __forceinline__ void dequant_tail_v32(const Gather &g, float rnorm, int row, int j,
                                                 uint32_t kr_base, int32_t *dbg) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {g.rp[i].x, g.rp[i].y, g.rp[i].z, g.rp[i].w};
    uint32_t f[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      f[k] = tc::pack_f16x2(__uint_as_float(w[k] << 16) * rnorm,
                            __uint_as_float(w[k] & 0xFFFF0000u) * rnorm);
    const uint32_t off = sw128_off(row, 0, 4 * j + i, 0);
    if (dbg_ok(dbg, off + 16u <= 16384u, kDbgSmemKv))
      tc::st_shared_v4(kr_base + off, f[0], f[1], f[2], f[3]);
  }
}

__device__ __forceinline__ int32_t load_sid(const Params &p, const Cursor &c, int row) {
  int32_t lid, row0;
  cursor_tile(p, c, lid, row0);
  const ListArgs &L = p.list[lid];
  const int32_t r = row0 + row;
  if (!dbg_ok(p.status, c.t >= 0 && c.t < p.T && r >= 0, kDbgIds)) return -1;
  return r < L.width ? __ldg(L.ids + (int64_t)c.t * L.idx_stride + r) : -1;
}

// Store of one 16-byte chunk into the 128 KiB KV tile (checked in the
// checking build).
__device__ __forceinline__ void st_kv(int32_t *dbg, uint32_t kv_base, uint32_t off, uint32_t a,
                                      uint32_t b, uint32_t c, uint32_t d) {
  if (dbg_ok(dbg, off + 16u <= 131072u, kDbgSmemKv)) tc::st_shared_v4(kv_base + off, a, b, c, d);
}

// Dequantize the two 64-dim k-blocks of M block mb for this thread's row.
__device__ __forceinline__ uint4 shfl_xor_u4(const uint4 v, int mask) {
  uint4 r;
  r.x = __shfl_xor_sync(0xffffffffu, v.x, mask);
  r.y = __shfl_xor_sync(0xffffffffu, v.y, mask);
  r.z = __shfl_xor_sync(0xffffffffu, v.z, mask);
  r.w = __shfl_xor_sync(0xffffffffu, v.w, mask);
  return r;
}

// Dequantize the two 64-dim k-blocks of M block mb for this thread's row
// half. Called by all 32 lanes of the warp (fp8 rows in sector layout get the
// missing half of each chunk pair from the other lane of their row).
__device__ __forceinline__ void dequant_block(bool fp8, bool ue, const Gather &g,
                                              const uint32_t (&scale2)[4], float rnorm, int mb,
                                              int row, int j, uint32_t kv_base, int32_t *dbg) {
  if (fp8) {
    // chunks c = 4m + 2j + e of k-block m; M block mb = k-blocks {2mb, 2mb+1}
#pragma unroll
    for (int mm = 0; mm < 2; ++mm) {
      const int m = 2 * mb + mm;
      const uint4 recv = shfl_xor_u4(j == 0 ? g.d[2 * m + 2] : g.d[2 * m], 1);
      const uint4 pr[2] = {g.pl ? g.d[2 * m] : g.d[2 * m + 1], g.pl ? g.d[2 * m + 1] : recv};
      // fp32 scales: scale2[mb] is the block's normalized f16 pair. ue8m0:
      // scale2 holds the 16 raw scale bytes; this lane's 32 dims of k-block m
      // (chunks 4m + 2j + e) take byte 2m + j, times the row's 2^-e (rnorm).
      const uint32_t sc =
          ue ? scale_f16x2(ue8m0_to_f32(scale2[m >> 1] >> (16 * (m & 1) + 8 * j)) * rnorm)
             : scale2[mb];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = 4 * m + 2 * j + e;   // dims [16c, 16c+16), scale block mb
        const uint32_t w[4] = {pr[e].x, pr[e].y, pr[e].z, pr[e].w};
        uint32_t f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tc::e4m3x4_to_f16x4(w[i], f[2 * i], f[2 * i + 1]);
          f[2 * i] = tc::hmul2(f[2 * i], sc);
          f[2 * i + 1] = tc::hmul2(f[2 * i + 1], sc);
        }
        const int ci = (2 * c) & 7;
        st_kv(dbg, kv_base, sw128_off(row, m, ci, 16384), f[0], f[1], f[2], f[3]);
        st_kv(dbg, kv_base, sw128_off(row, m, ci + 1, 16384), f[4], f[5], f[6], f[7]);
      }
    }
  } else {
    // chunk c = 4m + 2j + e holds dims [32c, 32c+32) of k-block 2m + j;
    // M block mb is m = mb, e in {0, 1}; its 4 scales are word 2mb + j of
    // the scale bytes (d[8] words 0..3, d[9] words 4..7). The two lanes of a
    // row write the same swizzle positions of two k-blocks; the odd lane
    // takes its halves in the other order (e = ee ^ j), so the 8 lanes of a
    // quarter-warp store to 8 different bank groups. Its chunk position
    // (4e + i) ^ (r % 8) is (4ee + i) ^ r7j with r7j = (r % 8) ^ 4j.
    const uint4 sq = mb < 2 ? g.d[8] : g.d[9];
    const uint32_t sw0 = j == 0 ? ((mb & 1) ? sq.z : sq.x) : ((mb & 1) ? sq.w : sq.y);
    const uint32_t sw = j == 0 ? sw0 : __funnelshift_l(sw0, sw0, 16);
    const uint32_t rb = (uint32_t)(2 * mb + j) * 16384u + (uint32_t)(row >> 3) * 1024u +
                        (uint32_t)(row & 7) * 128u;
    const int r7j = (row & 7) ^ (4 * j);
#pragma unroll
    for (int ee = 0; ee < 2; ++ee) {
      const uint4 src = (ee == j) ? g.d[2 * mb] : g.d[2 * mb + 1];
      const uint32_t pair = (sw >> (16 * ee)) & 0xFFFFu;
      const uint32_t s2 = tc::e4m3x2_to_f16x2(pair);
      const uint32_t sa = __byte_perm(s2, s2, 0x1010), sb = __byte_perm(s2, s2, 0x3232);
      const uint32_t w[4] = {src.x, src.y, src.z, src.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // word i = dims [32c + 8i, +8)
        uint32_t f[4];
        tc::e2m1x8_to_f16x8(w[i], f);
        const uint32_t sc = i < 2 ? sa : sb;
#pragma unroll
        for (int q = 0; q < 4; ++q) f[q] = tc::hmul2(f[q], sc);
        st_kv(dbg, kv_base, rb + ((uint32_t)((4 * ee + i) ^ r7j) << 4), f[0], f[1], f[2], f[3]);
      }
    }
  }
}

// MODEL1 rows (kM1): M block mb = k-blocks 2mb, 2mb+1. k-blocks 0..6 hold
// e4m3 codes times ue8m0 byte m (one per 64 dims; this lane's record chunks
// c = 2i + j, i = 2m, 2m+1), k-block 7 the bf16 RoPE dims (i = 14..17);
// every value times the row's 2^-e (rnorm), as f16. Called by all 32 lanes
// (the realignment trades halves between the two lanes of a row).
__device__ __forceinline__ uint4 model1_chunk(const Gather &g, int i, int j) {
  // off the grid: chunk 2i + j = A[2i+j].zw ++ A[2i+j+1].xy, where A[2i+j+1]
  // is the other lane's d[i] (j = 0) or d[i+1] (j = 1), and A[36].xy = tail.xy
  const uint4 send = (j == 0 && i < 17) ? g.d[i + 1] : g.d[i];
  const uint4 recv = shfl_xor_u4(send, 1);
  const uint4 nx = (j == 1 && i == 17) ? g.tail : recv;
  const uint4 own = g.d[i];
  return g.pl ? own : make_uint4(own.z, own.w, nx.x, nx.y);
}
__device__ __forceinline__ void dequant_block_model1(const Gather &g, float rnorm, int mb, int row,
                                                     int j, uint32_t kv_base, int32_t *dbg) {
#pragma unroll
  for (int mm = 0; mm < 2; ++mm) {
    const int m = 2 * mb + mm;
    if (m < 7) {
      const uint32_t sb = (m < 4 ? g.tail.z : g.tail.w) >> (8 * (m & 3));
      const uint32_t sc = scale_f16x2(ue8m0_to_f32(sb) * rnorm);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint4 src = model1_chunk(g, 2 * m + e, j);   // dims 64m + 16(2e + j) .. +16
        const uint32_t w[4] = {src.x, src.y, src.z, src.w};
        uint32_t f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tc::e4m3x4_to_f16x4(w[i], f[2 * i], f[2 * i + 1]);
          f[2 * i] = tc::hmul2(f[2 * i], sc);
          f[2 * i + 1] = tc::hmul2(f[2 * i + 1], sc);
        }
        const int ci = 2 * (2 * e + j);
        st_kv(dbg, kv_base, sw128_off(row, m, ci, 16384), f[0], f[1], f[2], f[3]);
        st_kv(dbg, kv_base, sw128_off(row, m, ci + 1, 16384), f[4], f[5], f[6], f[7]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {   // dims 448 + 8(2e + j) .. +8
        const uint4 src = model1_chunk(g, 14 + e, j);
        const uint32_t w[4] = {src.x, src.y, src.z, src.w};
        uint32_t f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          f[i] = tc::pack_f16x2(bf16_bits_to_f32(w[i] & 0xFFFFu) * rnorm,
                                bf16_bits_to_f32(w[i] >> 16) * rnorm);
        st_kv(dbg, kv_base, sw128_off(row, 7, 2 * e + j, 16384), f[0], f[1], f[2], f[3]);
      }
    }
  }
}

// Named barrier 1 among the 256 softmax threads (optionally OR-reducing).
__device__ __forceinline__ int sm_bar_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, 1, 256, p;\n\t"
      "selp.b32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred)
      : "memory");
  return r;
}
__device__ __forceinline__ void sm_bar() { asm volatile("barrier.cta.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar))
               : "memory");
}

// S = K . Q^T over the whole tile into TMEM (columns kColS..): the 32 MMAs
// (36 with the V3.2 tail tile) go out back to back from one thread, then a
// commit to `sfull`. The issue loop holds no waits or warp syncs: an
// mbarrier access of the issuing thread stalls its issue while earlier MMAs
// stream operands.
template <int HPG, bool kV32>
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint32_t kv_base, uint32_t q_base,
                                         uint32_t kr_base, uint64_t *sfull) {
  using Cfg = TcCfg<HPG, kV32>;
  const uint64_t dA = tc::sdesc(kv_base, 16, 1024, tc::kSwz128);
  const uint64_t dB = tc::sdesc(q_base, 16, 1024, tc::kSwz128);
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t ad = dA + (uint64_t)((kb * 16384 + ks * 32) >> 4);
      const uint64_t bd = dB + (uint64_t)((kb * HPG * 128 + ks * 32) >> 4);
      tc::mma_f16(tmem + Cfg::kColS, ad, bd, Cfg::kIdQK, (kb | ks) ? 1u : 0u);
    }
  }
  if constexpr (kV32) {   // key dims 512..575: the tail tile against Q's k-block 8
    const uint64_t dA_kr = tc::sdesc(kr_base, 16, 1024, tc::kSwz128);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_f16(tmem + Cfg::kColS, dA_kr + (uint64_t)((ks * 32) >> 4),
                  dB + (uint64_t)((8 * HPG * 128 + ks * 32) >> 4), Cfg::kIdQK, 1u);
  }
  tc::mma_commit(sfull);
}

// kExt: the V4.1 options (fp8 records with ue8m0 scales, GPT-J RoPE, MXFP8
// output); the plain instantiation compiles none of their code. kM1: MODEL1
// records as well, in instantiations of their own (with or without kExt).
// kStrict: the plan carries a wait budget (a test knob); only that
// instantiation compiles the exact-budget waits. kV32: V3.2 records (576-dim
// keys and Q: a 16 KB tile of the key dims 512..575 and a 9-block Q tile;
// at most 32 heads per group, no RoPE). kShared: several head groups read
// the same tiles (plain form); only group 0 prefetches records into L2.
// kPQ (plain form, for schedules with few tiles per token): the producers,
// idle at a token boundary once the next tile is written, stage the next
// token's Q and issue its first QK, which then overlap the softmax warps'
// finalize of the previous token. With many tiles per token the form
// without it is faster (its steady state measured about 1.5 % shorter).
template <int HPG, bool kExt, bool kStrict, bool kM1, bool kV32, bool kShared = false,
          bool kPQ = false>
__global__ void __launch_bounds__(kTcThreads, 1) tc_decode_kernel(Params p) {
  using Cfg = TcCfg<HPG, kV32>;
  constexpr int NH = Cfg::kHalf;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = tc::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  if (pad + Cfg::kBytes > Cfg::kSmem) {   // swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) report_status(p.status, DSA_ERR_UNSUPPORTED);
    return;
  }
  uint8_t *smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;
  const uint32_t kv_base = sbase + Cfg::kKV;
  const uint32_t q_base = sbase + Cfg::kQ;
  const uint32_t kr_base = sbase + Cfg::kKR;   // V3.2 records only
  const uint32_t p_base = sbase + Cfg::kP;
  int32_t *row_e_s = reinterpret_cast<int32_t *>(smem + Cfg::kRho);
  float *m_s = reinterpret_cast<float *>(smem + Cfg::kM);
  float *headf_s = reinterpret_cast<float *>(smem + Cfg::kHeadF);
  float *red_s = reinterpret_cast<float *>(smem + Cfg::kRed);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kMisc);
  volatile int32_t *abort_s = reinterpret_cast<volatile int32_t *>(smem + Cfg::kMisc + kMiscAbort);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kMisc + kMiscTmem);
  uint32_t *cnt_s = reinterpret_cast<uint32_t *>(smem + Cfg::kMisc + kMiscCnt);
  uint32_t *qk_cnt = reinterpret_cast<uint32_t *>(smem + Cfg::kMisc + kMiscQk);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hg = blockIdx.x % p.HG;
  const int cta = blockIdx.x / p.HG;
  const int h0 = hg * HPG;
  int64_t u0, u1;   // live-balanced unit range (the KV area is free scratch here)
  cta_range(p, cta, reinterpret_cast<int64_t *>(smem + Cfg::kKV), u0, u1);
  if (u0 >= u1) return;

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, Cfg::kCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b)
      tc::mbar_init(&bars[b], (b == kBarKvFull || b == kBarDrainQK) ? kPrWarps : 1u);
    tc::fence_mbar_init();
    *abort_s = 0;
    for (int i = 0; i < 8; ++i) cnt_s[i] = 0;
    *qk_cnt = 0;
  }
  if constexpr (kPQ) {   // the running max of the first token (finalize resets it after)
    if (tid < HPG) m_s[tid] = kMaxInit;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Bounded wait on a barrier phase. After any timeout (here or in another
  // warp) it returns at once; callers keep their control flow unchanged.
  // Waits off the MMA-issue path sleep between polls; the issuing warp spins.
  // A budget from the plan (a test knob, kStrict) is kept exactly: its polls
  // do not suspend (try_wait may suspend the thread for longer than a short
  // budget).
  auto wait = [&](int b, uint32_t &phase) {
    if (!*abort_s) {
      bool done;
      if constexpr (kStrict)
        done = tc::mbar_wait_strict(&bars[b], phase, p.wait_budget);
      else
        done = tc::mbar_wait(&bars[b], phase, kWaitBudget, warp == 0 ? 0u : 2000u);
      if (!done && !*abort_s) {
        *abort_s = 1;
        report_status(p.status, DSA_ERR_TIMEOUT);
      }
    }
    phase ^= 1u;
  };

  if (warp >= kSmWarps) {
    // ======================================================== producers
    tc::setmaxnreg_dec<Cfg::kPrRegs>();
    const int pw = warp - kSmWarps;
    // the two lanes of a row hold its two halves (j), so they can trade data
    const int row = 16 * pw + (lane >> 1), j = lane & 1;
    // kPQ: Q of token t -> f16 K-major SW128 tile, staged here once the
    // token's first tile is written (the previous token's last QK has read the old
    // Q by then: its PV blocks are free). RoPE in fp32 (NeoX or GPT-J), then
    // a power-of-two prescale per head so its max |q| lies in [1, 2): exact
    // for bf16 inputs whose exponents fit f16's range after scaling; the
    // factor goes to headf_s. Warp pw stages heads pw, pw + 8, ..., kQB at a
    // time (their loads issued together: one round trip per batch), each
    // rotated, reduced and stored without any cross-warp step.
    static_assert(HPG % kPrWarps == 0, "heads per producer warp");
    constexpr int kQH = HPG / kPrWarps;
    constexpr int kQB = kQH < 4 ? kQH : 4;
    auto stage_q_pr = [&](int32_t t) {
      int64_t pos = p.positions ? __ldg(p.positions + t) : 0;
      if (pos < 0 || (p.cos_sin && pos >= p.cs_rows)) {   // outside the table: flag, row 0
        if (pw == 0 && lane == 0) report_status(p.status, DSA_ERR_INVALID_ARG);
        pos = 0;
      }
      // Lane -> dims: lanes 0..27 hold 8-dim chunks 2 lane and 2 lane + 1
      // (dims 16 lane .. 16 lane + 15); lanes 28..31 (the RoPE dims
      // 448..511) hold chunks 56 + r and 60 + r, r = lane - 28 (dims
      // 448 + 8r .. +7 and 480 + 8r .. +7), so that both NeoX pairs
      // (448 + i, 480 + i) and GPT-J pairs (448 + 2i, 449 + 2i) lie inside
      // one lane and the rotation needs no shuffles.
      const bool rl = lane >= 28;
      const int ca = rl ? 56 + (lane - 28) : 2 * lane, cb = rl ? 60 + (lane - 28) : 2 * lane + 1;
      const bool rope = p.cos_sin != nullptr;
      const bool gptj = kExt && p.rope_gptj != 0;
      const bool rot = rope && rl && dbg_ok(p.status, pos >= 0 && pos < p.cs_rows, kDbgTable);
      // This lane's cos / sin from the token's table row: NeoX pairs
      // 8r .. 8r + 7; GPT-J pairs 4r .. 4r + 3 (chunk 56 + r) and
      // 16 + 4r .. 16 + 4r + 3 (chunk 60 + r). Entry i is cos, i + 32 sin.
      // Re-read (from L1) for every head rather than held in registers.
      const float4 *cs_row = rot ? reinterpret_cast<const float4 *>(p.cos_sin + pos * 64) : nullptr;
      const int f0 = gptj ? lane - 28 : 2 * (lane - 28), f1 = gptj ? lane - 24 : 2 * (lane - 28) + 1;
#pragma unroll 1
      for (int i0 = 0; i0 < kQH; i0 += kQB) {
        uint4 qa[kQB], qb[kQB];
        uint4 qc[kV32 ? kQB : 1];   // V3.2: lanes 0..7 also hold chunk 64 + lane (dims 512..575)
#pragma unroll
        for (int i = 0; i < kQB; ++i) {
          const int hq = h0 + pw + kPrWarps * (i0 + i);
          const __nv_bfloat16 *qh = p.q + (int64_t)t * p.q_st + (int64_t)hq * p.q_sh;
          if (dbg_ok(p.status, t >= 0 && t < p.T && hq < p.H, kDbgQ)) {
            qa[i] = __ldg(reinterpret_cast<const uint4 *>(qh) + ca);
            qb[i] = __ldg(reinterpret_cast<const uint4 *>(qh) + cb);
            if constexpr (kV32)
              qc[i] = lane < 8 ? __ldg(reinterpret_cast<const uint4 *>(qh) + 64 + lane)
                               : make_uint4(0, 0, 0, 0);
          } else {
            qa[i] = qb[i] = make_uint4(0, 0, 0, 0);
            if constexpr (kV32) qc[i] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int i = 0; i < kQB; ++i) {
          const int h = pw + kPrWarps * (i0 + i);
          const uint32_t w[8] = {qa[i].x, qa[i].y, qa[i].z, qa[i].w, qb[i].x, qb[i].y, qb[i].z, qb[i].w};
          float v[16];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            v[2 * k] = bf16_bits_to_f32(w[k] & 0xFFFFu);
            v[2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
          }
          if (rot) {
            const float4 ca0 = tc::ldg_f4_here(cs_row + f0), ca1 = tc::ldg_f4_here(cs_row + f1);
            const float4 sa0 = tc::ldg_f4_here(cs_row + 8 + f0), sa1 = tc::ldg_f4_here(cs_row + 8 + f1);
            const float c8[8] = {ca0.x, ca0.y, ca0.z, ca0.w, ca1.x, ca1.y, ca1.z, ca1.w};
            const float s8[8] = {sa0.x, sa0.y, sa0.z, sa0.w, sa1.x, sa1.y, sa1.z, sa1.w};
            if (gptj) {   // (v[2m], v[2m+1]) pair 4r + m; (v[8+2m], v[9+2m]) pair 16 + 4r + m
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                const int a = 2 * m;   // m < 4: chunk A, else chunk B (c8/s8 index m)
                const float x1 = v[a], x2 = v[a + 1];
                v[a] = fmaf(x1, c8[m], -(x2 * s8[m]));
                v[a + 1] = fmaf(x2, c8[m], x1 * s8[m]);
              }
            } else {      // (v[k], v[8+k]) pair 8r + k
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float x1 = v[k], x2 = v[8 + k];
                v[k] = fmaf(x1, c8[k], -(x2 * s8[k]));
                v[8 + k] = fmaf(x2, c8[k], x1 * s8[k]);
              }
            }
          }
          float mx = 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) mx = fmaxf(mx, fabsf(v[k]));
          float vc[8];   // V3.2: the lane's dims of chunk 64 + lane (zeros past lane 7)
          if constexpr (kV32) {
            const uint32_t wc[4] = {qc[i].x, qc[i].y, qc[i].z, qc[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              vc[2 * k] = bf16_bits_to_f32(wc[k] & 0xFFFFu);
              vc[2 * k + 1] = bf16_bits_to_f32(wc[k] >> 16);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf(vc[k]));
          }
          // max |q| of the head: non-negative floats order as their bits
          const uint32_t mbits = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
          int e = mbits ? (int)((mbits >> 23) & 0xFF) - 127 : 0;
          e = e < -126 ? -126 : (e > 126 ? 126 : e);
          const float down = __uint_as_float((uint32_t)(127 - e) << 23);
          if (lane == 0) headf_s[h] = p.scale_log2 * __uint_as_float((uint32_t)(127 + e) << 23);
          uint32_t f[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) f[k] = tc::pack_f16x2(v[2 * k] * down, v[2 * k + 1] * down);
          const uint32_t qo = sw128_off(h, ca >> 3, ca & 7, HPG * 128);
          const uint32_t qo1 = sw128_off(h, cb >> 3, cb & 7, HPG * 128);
          if (dbg_ok(p.status, qo + 16u <= HPG * 1024u && qo1 + 16u <= HPG * 1024u, kDbgSmemQ)) {
            tc::st_shared_v4(q_base + qo, f[0], f[1], f[2], f[3]);
            tc::st_shared_v4(q_base + qo1, f[4], f[5], f[6], f[7]);
          }
          if constexpr (kV32) {   // chunk 64 + lane into k-block 8
            if (lane < 8) {
              uint32_t fc[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) fc[k] = tc::pack_f16x2(vc[2 * k] * down, vc[2 * k + 1] * down);
              const uint32_t qo2 = sw128_off(h, 8, lane, HPG * 128);
              if (dbg_ok(p.status, qo2 + 16u <= HPG * 1152u, kDbgSmemQ))
                tc::st_shared_v4(q_base + qo2, fc[0], fc[1], fc[2], fc[3]);
            }
          }
        }
      }
    };
    uint32_t ph_free[4] = {0, 0, 0, 0};
    bool first = true;
    bool new_tok = true;   // kPQ: the tile opens a token, Q is staged with it
    int warm = 0;
    uint32_t kept = 0, chk = 0, pord = 0;
    // Tile records are loaded into registers one tile ahead, and prefetched
    // into L2 (bulk, one thread per row) two tiles ahead while the CTA warms
    // up and for fp8 tiles (see below).
    auto prefetch = [&](const Cursor &c, int32_t sid) {
      if (j != 0 || c.u >= u1) return;
      if constexpr (kShared) {   // the other groups' loads find the records in L2
        if (hg != 0) return;
      }
      int32_t lid2, row02;
      cursor_tile(p, c, lid2, row02);
      const ListArgs &L = p.list[lid2];
      if (slot_valid(L, row02 + row, lid2 == 0 ? c.lim0 : c.lim1, sid)) {
        const uint8_t *rec = record_ptr(L, sid);
        if (kM1 && L.fmt == DSA_REC_MODEL1_584) {   // 16-byte aligned span around the record
          const uintptr_t a0 = reinterpret_cast<uintptr_t>(rec) & ~(uintptr_t)15;
          const uintptr_t a1 = (reinterpret_cast<uintptr_t>(rec) + 584 + 15) & ~(uintptr_t)15;
          tc::prefetch_l2_bulk(reinterpret_cast<const void *>(a0), (uint32_t)(a1 - a0));
        } else {
          tc::prefetch_l2_bulk(rec, (uint32_t)L.rec);
        }
      }
    };
    Cursor cu = cursor_at(p, u0);       // tile being dequantized
    cursor_first_live(p, cu, u1);
    Cursor cn = cu;                     // next live tile
    if (cn.u < u1) cursor_next_live(p, cn, u1);
    int32_t sid_n1 = cn.u < u1 ? load_sid(p, cn, row) : -1;   // sid of the next tile
    Gather g;
    if (cu.u < u1) {
      const int32_t sid0 = load_sid(p, cu, row);
      prefetch(cu, sid0);
      prefetch(cn, sid_n1);
      issue_loads<kM1, kV32>(p, cu, sid0, row, j, g);
    }
    while (cu.u < u1) {
      const int32_t t = cu.t;
      int32_t lid, row0;
      cursor_tile(p, cu, lid, row0);
      Cursor cn2 = cn;
      if (cn2.u < u1) cursor_next_live(p, cn2, u1);
      const int32_t sid_n2 = cn2.u < u1 ? load_sid(p, cn2, row) : -1;
      const int32_t sid_next = sid_n1;
      const bool last_of_token = cn.u >= u1 || cn.t != t;
      const bool m1 = kM1 && p.list[lid].fmt == DSA_REC_MODEL1_584;
      const bool fp8 = !m1 && p.list[lid].fmt != DSA_REC_NVFP4_288;
      const bool ue = kExt && p.list[lid].fmt == DSA_REC_FP8_528_UE8M0;
      uint32_t scale2[4] = {0, 0, 0, 0};
      // Row exponent e (fp8 rows): the tile holds k * 2^-e, so the row's
      // largest block scale lies in [1, 2) and every block within 2^14 of it
      // keeps f16 precision, whatever the row's magnitude. NVFP4 rows (e2m1
      // times an e4m3 scale: exact f16 normals) keep e = 0.
      int erow = 0;
      if (fp8) {   // sector layout: lane j = 1 takes the scales from lane j = 0
        const uint4 sp = shfl_xor_u4(g.d[17], 1);
        const uint4 sv = (!g.pl && j == 1) ? sp : g.d[17];
        scale2[0] = sv.x;
        scale2[1] = sv.y;
        scale2[2] = sv.z;
        scale2[3] = sv.w;
        if (ue) {   // raw bytes, decoded per k-block; e from the largest byte
          uint32_t mx = __vmaxu4(__vmaxu4(sv.x, sv.y), __vmaxu4(sv.z, sv.w));
          mx = max(max(mx & 0xFFu, (mx >> 8) & 0xFFu), max((mx >> 16) & 0xFFu, mx >> 24));
          erow = row_exp(mx);
        } else {    // e from the largest exponent field of the 4 fp32 scales
          const uint32_t f = max(max((sv.x >> 23) & 0xFFu, (sv.y >> 23) & 0xFFu),
                                 max((sv.z >> 23) & 0xFFu, (sv.w >> 23) & 0xFFu));
          int fe = (int)f;
          if constexpr (kV32) {
            // and from the bf16 key dims' largest magnitude (exponent field
            // minus 8, as for MODEL1), over both halves of the row
            uint32_t bm = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              bm = __vmaxu2(bm, __vmaxu2(__vmaxu2(g.rp[i].x & 0x7FFF7FFFu, g.rp[i].y & 0x7FFF7FFFu),
                                         __vmaxu2(g.rp[i].z & 0x7FFF7FFFu, g.rp[i].w & 0x7FFF7FFFu)));
            bm = max(bm & 0xFFFFu, bm >> 16);
            bm = max(bm, (uint32_t)__shfl_xor_sync(0xffffffffu, bm, 1));
            fe = max(fe, (int)(bm >> 7) - 8);
          }
          erow = row_exp((uint32_t)max(fe, 0));
          const float rn = pow2i(-erow);
#pragma unroll
          for (int b = 0; b < 4; ++b) scale2[b] = scale_f16x2(__uint_as_float(scale2[b]) * rn);
        }
      }
      if (m1) {
        // e from the largest scale byte and from the bf16 part's largest
        // magnitude (its exponent field minus 8), so the f16 values stay
        // below 2^9 either way. The bf16 words: tail.xy and d[14..17], except
        // that off the grid lane 0's d[14] starts 8 bytes early (fp8 codes).
        uint32_t mx = __vmaxu4(g.tail.z, g.tail.w & 0x00FFFFFFu);
        mx = max(max(mx & 0xFFu, (mx >> 8) & 0xFFu), max((mx >> 16) & 0xFFu, mx >> 24));
        uint32_t bm = __vmaxu2(g.tail.x & 0x7FFF7FFFu, g.tail.y & 0x7FFF7FFFu);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = g.d[14 + q];
          const bool lo_fp8 = q == 0 && !g.pl && j == 0;
          const uint32_t vx = lo_fp8 ? 0u : v.x, vy = lo_fp8 ? 0u : v.y;
          bm = __vmaxu2(bm, __vmaxu2(__vmaxu2(vx & 0x7FFF7FFFu, vy & 0x7FFF7FFFu),
                                     __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
        }
        bm = max(bm & 0xFFFFu, bm >> 16);
        bm = max(bm, (uint32_t)__shfl_xor_sync(0xffffffffu, bm, 1));   // the row's other half
        const int eb = (int)(bm >> 7) - 8;   // bf16 exponent field - 8 (biased)
        erow = row_exp(max((int)mx, eb));
      }
      const float rnorm = pow2i(-erow);
      if (j == 0 && g.ok) {
        kept += 1;
        chk += row_hash(g.sid, g.r, lid);
      }
      if (last_of_token) {   // add this warp's kept-row record of token t to its slot
        uint32_t k2 = kept, c2 = chk;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          k2 += __shfl_xor_sync(0xffffffffu, k2, off);
          c2 += __shfl_xor_sync(0xffffffffu, c2, off);
        }
        if (lane == 0) {
          atomicAdd(&cnt_s[(pord & 3) * 2], k2);
          atomicAdd(&cnt_s[(pord & 3) * 2 + 1], c2);
        }
        kept = 0;
        chk = 0;
        ++pord;
      }
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
        if (!first) wait(kBarKvFree + mb, ph_free[mb]);
        if (mb == 0 && j == 0) row_e_s[row] = g.ok ? erow : kRowInvalid;
        if (m1)
          dequant_block_model1(g, rnorm, mb, row, j, kv_base, p.status);
        else
          dequant_block(fp8, ue, g, scale2, rnorm, mb, row, j, kv_base, p.status);
        if constexpr (kV32) {   // key dims 512..575 once the previous QK has read them
          if (mb == 0) dequant_tail_v32(g, rnorm, row, j, kr_base, p.status);
        }
      }
      const bool opens = kPQ && new_tok;   // the token's first tile in this CTA
      if constexpr (kPQ) {
        if (opens) {
          // The next tile's loads rewrite only part of g (by format and
          // lane): clearing it here keeps the rest from being held in
          // registers through the staging.
          g = Gather{};
          stage_q_pr(t);
        }
        new_tok = last_of_token;
      }
      // One hand-off per tile: the QK MMAs are issued once the whole tile is
      // in place, so per-block fences and arrives would only lengthen the
      // dequant chain.
      tc::fence_async_smem();
      __syncwarp();
      if constexpr (kPQ) {
        if (lane == 0) {
          mbar_arrive(&bars[kBarKvFull]);
          // A token's first QK goes out from here, so that it runs while the
          // softmax warps finalize the previous token: from lane 0 of the
          // producer warp that lands its rows last (an acquire-release count
          // of the warps done tells it, with no wait).
          if (opens && (tc::atom_add_acq_rel_shared(qk_cnt, 1u) & (kPrWarps - 1)) == kPrWarps - 1 &&
              !*abort_s) {
            tc::tc_fence_after();
            issue_qk<HPG, kV32>(tmem, kv_base, q_base, kr_base, &bars[kBarSFull]);
          }
        }
      } else {
        if (lane == 0) mbar_arrive(&bars[kBarKvFull]);
      }
      first = false;
      // L2 prefetch two tiles ahead: while the CTA warms up, and always for
      // fp8 tiles, whose 17 sector loads per row otherwise keep the load
      // queue full into the softmax (config 4: +7 %); for NVFP4 tiles the
      // register loads alone cover the latency (prefetching them cost 1.5 %).
      if (warm < 2 || p.list[cn2.k < p.list[0].tiles ? 0 : 1].fmt != DSA_REC_NVFP4_288)
        prefetch(cn2, sid_n2);
      ++warm;
      cu = cn;
      cn = cn2;
      sid_n1 = sid_n2;
      if (cu.u < u1) issue_loads<kM1, kV32>(p, cu, sid_next, row, j, g);
    }
  } else {
    // ======================================================== softmax / epilogue / MMA
    tc::setmaxnreg_inc<Cfg::kSmRegs>();
    const int q4 = warp & 3, half = warp >> 2;
    const int prow = 32 * q4 + lane;
    const uint32_t tl_lane = tmem + ((uint32_t)(32 * q4) << 16);
    const bool issuer = tid == 0;   // issues every tcgen05.mma and commit
    // Descriptor bases; an offset of `o` bytes adds o >> 4 to the start
    // address field (no carry: shared addresses stay below 256 KiB).
    const uint64_t dA_qk = tc::sdesc(kv_base, 16, 1024, tc::kSwz128);
    const uint64_t dB_qk = tc::sdesc(q_base, 16, 1024, tc::kSwz128);
    const uint64_t dA_pv = tc::sdesc(kv_base, 16384, 1024, tc::kSwz128);
    const uint64_t dB_pv = tc::sdesc(p_base, Cfg::kPBytes, 8 * Cfg::kPRow, Cfg::kPSwz);
    uint32_t ph_s = 0, ph_kv = 0, ph_of = 0, sord = 0;
    float l_reg[NH];              // per-head partial sums of this row
    const float4 *m_s4 = reinterpret_cast<const float4 *>(m_s) + half * (NH / 4);
    // per head: scale * log2(e) * 2^e, e the exponent of the head's Q prescale
    const float4 *hf_s4 = reinterpret_cast<const float4 *>(headf_s) + half * (NH / 4);
    bool seg_worked = false, first_pv = true;
    // the sink logit of head tid, read once (finalize needs it per token)
    const float sink_h = (tid < HPG && p.sink) ? __ldg(p.sink + h0 + tid) : 0.f;

    // Q of token t -> f16 K-major SW128 tile. RoPE (NeoX) in fp32, then a
    // power-of-two prescale per head so its max |q| lies in [1, 2): exact
    // for bf16 inputs whose exponents fit f16's range after scaling; the
    // factor goes to headf_s. Each warp stages heads warp, warp + 8, ...:
    // all their loads are issued first (one round trip), then each head is
    // rotated, reduced and stored without any cross-warp step.
    static_assert(HPG % kSmWarps == 0, "heads per softmax warp");
    constexpr int kQH = HPG / kSmWarps;
    auto stage_q = [&](int32_t t) {
      int64_t pos = p.positions ? __ldg(p.positions + t) : 0;
      if (pos < 0 || (p.cos_sin && pos >= p.cs_rows)) {   // outside the table: flag, row 0
        if (tid == 0) report_status(p.status, DSA_ERR_INVALID_ARG);
        pos = 0;
      }
      // Lane -> dims: lanes 0..27 hold 8-dim chunks 2 lane and 2 lane + 1
      // (dims 16 lane .. 16 lane + 15); lanes 28..31 (the RoPE dims
      // 448..511) hold chunks 56 + r and 60 + r, r = lane - 28 (dims
      // 448 + 8r .. +7 and 480 + 8r .. +7), so that both NeoX pairs
      // (448 + i, 480 + i) and GPT-J pairs (448 + 2i, 449 + 2i) lie inside
      // one lane and the rotation needs no shuffles.
      const bool rl = lane >= 28;
      const int ca = rl ? 56 + (lane - 28) : 2 * lane, cb = rl ? 60 + (lane - 28) : 2 * lane + 1;
      uint4 qa[kQH], qb[kQH];
      uint4 qc[kV32 ? kQH : 1];   // V3.2: lanes 0..7 also hold chunk 64 + lane (dims 512..575)
#pragma unroll
      for (int i = 0; i < kQH; ++i) {
        const int hq = h0 + warp + kSmWarps * i;
        const __nv_bfloat16 *qh = p.q + (int64_t)t * p.q_st + (int64_t)hq * p.q_sh;
        if (dbg_ok(p.status, t >= 0 && t < p.T && hq < p.H, kDbgQ)) {
          qa[i] = __ldg(reinterpret_cast<const uint4 *>(qh) + ca);
          qb[i] = __ldg(reinterpret_cast<const uint4 *>(qh) + cb);
          if constexpr (kV32)
            qc[i] = lane < 8 ? __ldg(reinterpret_cast<const uint4 *>(qh) + 64 + lane)
                             : make_uint4(0, 0, 0, 0);
        } else {
          qa[i] = qb[i] = make_uint4(0, 0, 0, 0);
          if constexpr (kV32) qc[i] = make_uint4(0, 0, 0, 0);
        }
      }
      // This lane's cos / sin from the token's table row: NeoX pairs
      // 8r .. 8r + 7; GPT-J pairs 4r .. 4r + 3 (chunk 56 + r) and
      // 16 + 4r .. 16 + 4r + 3 (chunk 60 + r). Entry i is cos, i + 32 sin.
      const bool rope = p.cos_sin != nullptr;
      const bool gptj = kExt && p.rope_gptj != 0;
      float c8[8], s8[8];
      if (rope && rl && dbg_ok(p.status, pos >= 0 && pos < p.cs_rows, kDbgTable)) {
        const float4 *row = reinterpret_cast<const float4 *>(p.cos_sin + pos * 64);
        const int r = lane - 28;
        const int f0 = gptj ? r : 2 * r, f1 = gptj ? 4 + r : 2 * r + 1;   // float4 index of cos
        const float4 ca0 = __ldg(row + f0), ca1 = __ldg(row + f1);
        const float4 sa0 = __ldg(row + 8 + f0), sa1 = __ldg(row + 8 + f1);
        c8[0] = ca0.x; c8[1] = ca0.y; c8[2] = ca0.z; c8[3] = ca0.w;
        c8[4] = ca1.x; c8[5] = ca1.y; c8[6] = ca1.z; c8[7] = ca1.w;
        s8[0] = sa0.x; s8[1] = sa0.y; s8[2] = sa0.z; s8[3] = sa0.w;
        s8[4] = sa1.x; s8[5] = sa1.y; s8[6] = sa1.z; s8[7] = sa1.w;
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          c8[k] = 1.f;
          s8[k] = 0.f;
        }
      }
      const bool rot = rope && rl;
#pragma unroll
      for (int i = 0; i < kQH; ++i) {
        const int h = warp + kSmWarps * i;
        const uint32_t w[8] = {qa[i].x, qa[i].y, qa[i].z, qa[i].w, qb[i].x, qb[i].y, qb[i].z, qb[i].w};
        float v[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          v[2 * k] = bf16_bits_to_f32(w[k] & 0xFFFFu);
          v[2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
        }
        if (rot) {
          if (gptj) {   // (v[2m], v[2m+1]) pair 4r + m; (v[8+2m], v[9+2m]) pair 16 + 4r + m
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const int a = 2 * m;   // m < 4: chunk A, else chunk B (c8/s8 index m)
              const float x1 = v[a], x2 = v[a + 1];
              v[a] = fmaf(x1, c8[m], -(x2 * s8[m]));
              v[a + 1] = fmaf(x2, c8[m], x1 * s8[m]);
            }
          } else {      // (v[k], v[8+k]) pair 8r + k
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float x1 = v[k], x2 = v[8 + k];
              v[k] = fmaf(x1, c8[k], -(x2 * s8[k]));
              v[8 + k] = fmaf(x2, c8[k], x1 * s8[k]);
            }
          }
        }
        float mx = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) mx = fmaxf(mx, fabsf(v[k]));
        float vc[8];   // V3.2: the lane's dims of chunk 64 + lane (zeros past lane 7)
        if constexpr (kV32) {
          const uint32_t wc[4] = {qc[i].x, qc[i].y, qc[i].z, qc[i].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            vc[2 * k] = bf16_bits_to_f32(wc[k] & 0xFFFFu);
            vc[2 * k + 1] = bf16_bits_to_f32(wc[k] >> 16);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf(vc[k]));
        }
        // max |q| of the head: non-negative floats order as their bits
        const uint32_t mbits = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
        int e = mbits ? (int)((mbits >> 23) & 0xFF) - 127 : 0;
        e = e < -126 ? -126 : (e > 126 ? 126 : e);
        const float down = __uint_as_float((uint32_t)(127 - e) << 23);
        if (lane == 0) headf_s[h] = p.scale_log2 * __uint_as_float((uint32_t)(127 + e) << 23);
        uint32_t f[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = tc::pack_f16x2(v[2 * k] * down, v[2 * k + 1] * down);
        const uint32_t qo = sw128_off(h, ca >> 3, ca & 7, HPG * 128);
        const uint32_t qo1 = sw128_off(h, cb >> 3, cb & 7, HPG * 128);
        if (dbg_ok(p.status, qo + 16u <= HPG * 1024u && qo1 + 16u <= HPG * 1024u, kDbgSmemQ)) {
          tc::st_shared_v4(q_base + qo, f[0], f[1], f[2], f[3]);
          tc::st_shared_v4(q_base + qo1, f[4], f[5], f[6], f[7]);
        }
        if constexpr (kV32) {   // chunk 64 + lane into k-block 8
          if (lane < 8) {
            uint32_t fc[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) fc[k] = tc::pack_f16x2(vc[2 * k] * down, vc[2 * k + 1] * down);
            const uint32_t qo2 = sw128_off(h, 8, lane, HPG * 128);
            if (dbg_ok(p.status, qo2 + 16u <= HPG * 1152u, kDbgSmemQ))
              tc::st_shared_v4(q_base + qo2, fc[0], fc[1], fc[2], fc[3]);
          }
        }
      }
      if (tid < HPG) m_s[tid] = kMaxInit;
      tc::fence_async_smem();
      sm_bar();   // Q (async proxy), head factors and m_s visible
    };

    // Split token t, merged in the run by the CTA that completed its units
    // (the combine kernel's arithmetic, parts in CTA order, so the result
    // does not depend on which CTA merges): parts are the CTAs c0..c1 whose
    // ranges meet the token's units [ts, te) -- every one of them has
    // arrived, and each wrote both ends of its range to p.bounds before its
    // partial. M = max_i lse_i, w_i = e^{lse_i - M}, out = sum_i w_i O_i /
    // (sum_i w_i + e^{sink - M}), lse = M + log sum_i w_i. The weights sit
    // in the P buffer (free between a token's last PV and the next
    // token's first softmax): at most 64 parts (the plan's condition).
    auto merge_token = [&](int32_t t) {
      const int64_t ts = (int64_t)t * p.tpt, te = ts + p.tpt;
      const long long *bnd = reinterpret_cast<const long long *>(p.bounds);
      int32_t *info = reinterpret_cast<int32_t *>(red_s + 128);   // c0, c1, c0 late
      if (warp == 0) {
        // The range starts around this CTA in one round trip (lane: CTA
        // cta - 16 + lane): c0 = the last CTA at or before this one whose
        // range starts at or before ts, c1 + 1 = the first after it whose
        // range starts at or past te. Lanes beyond the parts may read ends
        // that CTAs not involved have not written yet; the ballots take
        // the bit nearest this CTA, which lies among the parts. A token
        // spanning beyond the window walks on from its edge.
        const int cb = cta - 16 + lane;
        const long long bv = (cb >= 0 && cb <= p.C) ? __ldcg(bnd + cb) : 0;
        const unsigned le = __ballot_sync(0xffffffffu, cb >= 0 && cb <= cta && bv <= ts);
        const unsigned ge = __ballot_sync(0xffffffffu, cb > cta && cb <= p.C && bv >= te);
        if (lane == 0) {
          int32_t c0 = le ? cta - 16 + (31 - __clz(le)) : cta - 16;
          int32_t c1 = ge ? cta - 16 + (__ffs(ge) - 1) - 1 : cta + 15;
          if (!le)
            while (c0 > 0 && __ldcg(bnd + c0) > ts) --c0;
          if (!ge)
            while (c1 + 1 < p.C && __ldcg(bnd + c1 + 1) < te) ++c1;
          c0 = c0 < 0 ? 0 : c0;
          c1 = c1 > p.C - 1 ? p.C - 1 : c1;
          info[0] = c0;
          info[1] = c1;
          info[2] = __ldcg(bnd + c0) < ts ? 1 : 0;
        }
      }
      sm_bar();
      const int32_t c0 = info[0], c1 = info[1];
      const bool c0_late = info[2] != 0;
      // partial slot of part c: 2c when t is the CTA's first token, else 2c + 1
      auto slot_of = [&](int32_t c) -> int64_t {
        return 2 * (int64_t)c + ((c == c0 && c0_late) ? 1 : 0);
      };
      int np = c1 - c0 + 1;   // >= 1; at most 64 by the plan, held here in every build
      if (np > 64) {
        if (tid == 0) report_status(p.status, DSA_ERR_UNSUPPORTED);
        np = 0;
      }
      const int64_t sb = (int64_t)hg * 2 * p.C;
      const int64_t part_n = (int64_t)p.HG * 2 * p.C * HPG;
      float *w_s = reinterpret_cast<float *>(smem + Cfg::kP);   // [np][HPG]
      // the parts' lse, one load per thread and round
      for (int e = tid; e < np * HPG; e += 256) {
        const int q = e / HPG, h = e - q * HPG;
        const int64_t ip = (sb + slot_of(c0 + q)) * HPG + h;
        w_s[e] = dbg_ok(p.status, ip >= 0 && ip < part_n, kDbgPartial) ? __ldcg(p.part_lse + ip)
                                                                     : -INFINITY;
      }
      if (warp == 2 && hg == 0) {   // row-selection record: lanes over the parts
        uint32_t k = 0, s2 = 0;
        for (int q = lane; q < np; q += 32) {
          const int64_t sl = slot_of(c0 + q);
          if (!dbg_ok(p.status, sl >= 0 && sl < 2 * p.C, kDbgSel)) continue;
          k += (uint32_t)__ldcg(p.part_sel + 2 * sl);
          s2 += (uint32_t)__ldcg(p.part_sel + 2 * sl + 1);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          k += __shfl_xor_sync(0xffffffffu, k, off);
          s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        }
        if (lane == 0 && dbg_ok(p.status, t >= 0 && t < p.T, kDbgSel)) {
          p.sel[2 * (int64_t)t] = (int32_t)k;
          p.sel[2 * (int64_t)t + 1] = (int32_t)s2;
        }
      }
      sm_bar();
      if (tid < HPG) {   // weights of head tid: M = max_q lse_q, w_q = e^{lse_q - M}
        const int h = tid;
        float mx = -INFINITY;
        for (int q = 0; q < np; ++q) mx = fmaxf(mx, w_s[q * HPG + h]);
        float z = 0.f;
        for (int q = 0; q < np; ++q) {
          const float li = w_s[q * HPG + h];
          const float w = (li == -INFINITY) ? 0.f : expf(li - mx);
          w_s[q * HPG + h] = w;
          z += w;
        }
        float inv = 0.f;
        if (z > 0.f) {
          float den = z;
          if (p.sink) den = (sink_h == INFINITY) ? INFINITY : z + expf(sink_h - mx);
          inv = 1.f / den;
        }
        red_s[h] = inv;
        const int64_t il = (int64_t)t * p.H + h0 + h;
        if (dbg_ok(p.status, il >= 0 && il < (int64_t)p.T * p.H, kDbgOut))
          p.lse[il] = (z > 0.f) ? mx + logf(z) : -INFINITY;
      }
      sm_bar();
      // out = sum_i w_i O_i * inv: thread items e = tid + 256 k, head
      // e / 128, float4 e % 128 of it; 8 items at a time, two parts' loads
      // in flight together.
      constexpr int kItems = HPG * (kD / 4) / 256;
      static_assert(kItems % 8 == 0, "merge items per thread");
      const float4 *po = reinterpret_cast<const float4 *>(p.part_o);
      float *const stage = kExt ? p.stage : nullptr;
#pragma unroll 1
      for (int k0 = 0; k0 < kItems; k0 += 8) {
        float4 acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int q = 0; q < np; q += 2) {
          const bool two = q + 1 < np;
          const int64_t s0 = (sb + slot_of(c0 + q)) * HPG;
          const int64_t s1 = two ? (sb + slot_of(c0 + q + 1)) * HPG : s0;
          float4 o0[8], o1[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int e = tid + 256 * (k0 + i), h = e >> 7, d4 = e & 127;
            const bool ok0 = dbg_ok(p.status, s0 + h >= 0 && s0 + h < part_n, kDbgPartial);
            const bool ok1 = dbg_ok(p.status, s1 + h >= 0 && s1 + h < part_n, kDbgPartial);
            o0[i] = ok0 ? __ldcg(po + (s0 + h) * (kD / 4) + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
            o1[i] = (two && ok1) ? __ldcg(po + (s1 + h) * (kD / 4) + d4)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int h = (tid + 256 * (k0 + i)) >> 7;
            const float w0 = w_s[q * HPG + h], w1 = two ? w_s[(q + 1) * HPG + h] : 0.f;
            acc[i].x = fmaf(w1, o1[i].x, fmaf(w0, o0[i].x, acc[i].x));
            acc[i].y = fmaf(w1, o1[i].y, fmaf(w0, o0[i].y, acc[i].y));
            acc[i].z = fmaf(w1, o1[i].z, fmaf(w0, o0[i].z, acc[i].z));
            acc[i].w = fmaf(w1, o1[i].w, fmaf(w0, o0[i].w, acc[i].w));
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = tid + 256 * (k0 + i), h = e >> 7, d4 = e & 127;
          const float inv = red_s[h];
          const int64_t io = ((int64_t)t * p.H + h0 + h) * kD + 4 * d4;
          if (!dbg_ok(p.status, io >= 0 && io + 4 <= (int64_t)p.T * p.H * kD, kDbgOut)) continue;
          if (stage != nullptr) {   // MXFP8 output: fp32 to the staging area, cast later
            *reinterpret_cast<float4 *>(stage + io) =
                make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv);
            continue;
          }
          const __nv_bfloat162 a = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
          const __nv_bfloat162 b = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t *>(&a);
          pk.y = *reinterpret_cast<const uint32_t *>(&b);
          *reinterpret_cast<uint2 *>(p.out + io) = pk;
        }
      }
      sm_bar();   // weights and red_s free again
    };

    // Token finished: sums over rows, sink, out / lse (or partial), selection.
    auto finalize = [&](const Segment &seg) {
      if (seg_worked) wait(kBarOFinal, ph_of);
      tc::tc_fence_after();
      // Sums over the warp's 32 rows, in place (l_reg restarts at zero with
      // the next token; it is all zeros when no tile was worked): recursive
      // halving -- at step st a lane keeps the upper half of its 2*st values
      // when lane bit st is set, else the lower half, and adds the partner's
      // copy of that half -- leaves head j's sum in lane j (NH < 32: lanes j,
      // j + NH, ... hold parts, folded by the last shuffles).
#pragma unroll
      for (int st = NH / 2; st >= 1; st >>= 1) {
        const bool up = (lane & st) != 0;
#pragma unroll
        for (int i = 0; i < st; ++i) {
          const float send = up ? l_reg[i] : l_reg[i + st];
          const float keep = up ? l_reg[i + st] : l_reg[i];
          l_reg[i] = keep + __shfl_xor_sync(0xffffffffu, send, st);
        }
      }
#pragma unroll
      for (int off = NH; off < 32; off <<= 1) l_reg[0] += __shfl_xor_sync(0xffffffffu, l_reg[0], off);
      if (lane < NH) red_s[q4 * 64 + half * NH + lane] = l_reg[0];
      sm_bar();
      if (tid < HPG) {   // 1 / denominator of head tid, lse
        const int h = tid;
        const float l = red_s[h] + red_s[64 + h] + red_s[128 + h] + red_s[192 + h];
        const float m = seg_worked ? m_s[h] : -INFINITY;
        if constexpr (kPQ) m_s[h] = kMaxInit;   // the next token's (ordered by the barrier below)
        float iv = 0.f;
        if (l > 0.f) {
          float den = l;
          if (seg.whole && p.sink) {
            const float sk = sink_h;
            den = (sk == INFINITY) ? INFINITY : l + tc::ex2(sk * kLog2e - m);
          }
          iv = 1.f / den;
        }
        const float lse = (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
        if (seg.whole) {
          const int64_t i = (int64_t)seg.t * p.H + h0 + h;
          if (dbg_ok(p.status, i >= 0 && i < (int64_t)p.T * p.H, kDbgOut)) p.lse[i] = lse;
        } else {
          const int64_t i = ((int64_t)hg * 2 * p.C + seg.slot) * HPG + h;
          if (dbg_ok(p.status, i >= 0 && i < (int64_t)p.HG * 2 * p.C * HPG, kDbgPartial))
            p.part_lse[i] = lse;
        }
        red_s[256 - 64 + h] = iv;   // read below; sums of row 3 were consumed above
      }
      if (tid == 0) {   // kept rows / checksum of the token, then clear the slot
        uint32_t k2 = 0, c2 = 0;
        if (seg_worked) {
          k2 = cnt_s[(sord & 3) * 2];
          c2 = cnt_s[(sord & 3) * 2 + 1];
          cnt_s[(sord & 3) * 2] = 0;
          cnt_s[(sord & 3) * 2 + 1] = 0;
        }
        if (hg == 0) {
          int32_t *dst =
              seg.whole ? (p.sel + 2 * (int64_t)seg.t) : (p.part_sel + 2 * (int64_t)seg.slot);
          if (dbg_ok(p.status, seg.whole ? (seg.t >= 0 && seg.t < p.T)
                                         : (seg.slot >= 0 && seg.slot < 2 * p.C), kDbgSel)) {
            dst[0] = (int32_t)k2;
            dst[1] = (int32_t)c2;
          }
        }
      }
      if (seg_worked) ++sord;
      sm_bar();
      // MXFP8 output: whole tokens go to the fp32 staging area (cast later)
      float *const stage = kExt ? p.stage : nullptr;
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
        const int d = 128 * mb + prow;
#pragma unroll
        for (int g8 = 0; g8 < NH / 8; ++g8) {
          float o[8];
          if (seg_worked) tc::tmem_ld<8>(tl_lane + Cfg::kColO + mb * HPG + half * NH + 8 * g8, o);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int h = half * NH + 8 * g8 + i;
            const float iv = red_s[256 - 64 + h];
            const float v = (!seg_worked || iv == 0.f) ? 0.f : o[i] * iv;
            const int64_t io = ((int64_t)seg.t * p.H + h0 + h) * kD + d;
            const int64_t ip = (((int64_t)hg * 2 * p.C + seg.slot) * HPG + h) * kD + d;
            if (seg.whole && !dbg_ok(p.status, io >= 0 && io < (int64_t)p.T * p.H * kD, kDbgOut))
              continue;
            if (!seg.whole &&
                !dbg_ok(p.status, ip >= 0 && ip < (int64_t)p.HG * 2 * p.C * HPG * kD, kDbgPartial))
              continue;
            if (seg.whole && stage != nullptr)
              stage[io] = v;
            else if (seg.whole)
              p.out[io] = __float2bfloat16_rn(v);
            else
              p.part_o[ip] = v;
          }
        }
      }
      tc::tc_fence_before();
      sm_bar();   // O read out (next PV may overwrite it); red_s free again
      if (p.merge && !seg.whole) {
        // Split token: count this part's units; the part that completes the
        // token merges it. Every thread's partial stores are fenced before
        // the count, the merging CTA fences again before reading the parts.
        __threadfence();
        int last = 0;
        if (tid == 0) {
          const int32_t units = (int32_t)(seg.u_end - seg.u_begin);
          const int64_t ic = (int64_t)hg * p.T + seg.t;
          if (dbg_ok(p.status, ic >= 0 && ic < (int64_t)p.HG * p.T, kDbgPartial))
            last = atomicAdd(p.tok_cnt + ic, units) + units == p.tpt;
        }
        if (sm_bar_or(last)) {
          __threadfence();
          merge_token(seg.t);
        }
      }
    };

    // One pass per token segment of the range: set-up, its tiles, then
    // finalize (the per-token work stays outside the tile loop).
    Cursor cu = cursor_at(p, u0);
    while (cu.u < u1) {
      const int32_t t = cu.t;
      const Segment seg = make_segment(p, cta, t, u0, u1);
      seg_worked = false;
      first_pv = true;
#pragma unroll
      for (int j = 0; j < NH; ++j) l_reg[j] = 0.f;
      if constexpr (!kPQ) {   // (kPQ: the producers stage it)
        // Q is staged only for tokens with a live tile in this range.
        Cursor cv = cu;
        cursor_first_live(p, cv, seg.u_end);
        if (cv.u < seg.u_end) stage_q(t);
      }
      for (; cu.u < u1 && cu.t == t; cursor_step(p, cu)) {
        if (!cursor_live(p, cu)) continue;
        seg_worked = true;
        // ---- S = K . Q^T over the whole tile: the MMAs go out back to back
        // once the producers have landed all of it, which keeps the issue
        // loop free of waits and warp syncs (an mbarrier access of the issuing
        // thread stalls its issue while earlier MMAs stream operands).
        // (kPQ: a token's first QK comes from the producers.)
        if (warp == 0) {
          wait(kBarKvFull, ph_kv);
          tc::tc_fence_after();
          if (issuer && !(kPQ && first_pv) && !*abort_s) {
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
              const uint32_t d_tmem = tmem + Cfg::kColS;
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ad = dA_qk + (uint64_t)((kb * 16384 + ks * 32) >> 4);
                const uint64_t bd = dB_qk + (uint64_t)((kb * HPG * 128 + ks * 32) >> 4);
                tc::mma_f16(d_tmem, ad, bd, Cfg::kIdQK, (kb | ks) ? 1u : 0u);
              }
            }
            if constexpr (kV32) {   // key dims 512..575: the tail tile against Q's k-block 8
              const uint64_t dA_kr = tc::sdesc(kr_base, 16, 1024, tc::kSwz128);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                tc::mma_f16(tmem + Cfg::kColS, dA_kr + (uint64_t)((ks * 32) >> 4),
                            dB_qk + (uint64_t)((8 * HPG * 128 + ks * 32) >> 4), Cfg::kIdQK, 1u);
            }
            tc::mma_commit(&bars[kBarSFull]);
          }
          __syncwarp();
        } else {
          // the row flags are written with block 0 of the tile
          wait(kBarKvFull, ph_kv);
        }
        // This thread's row: kept or not, and its exponent e (the tile holds
        // k * 2^-e). In log2 units the row's score is x = S * hf * 2^e; the
        // running max m and P work on y = x + e, so P = 2^(y - m) carries the
        // factor 2^e that PV needs to rebuild k from the tile, while the row
        // sums take P * 2^-e = 2^(x - m): out = O / l and lse = m + log2 l
        // keep their form. Rows that are not kept get y = -inf (P = 0).
        const int32_t ei = row_e_s[prow];
        const bool rv = ei != kRowInvalid;
        const float er = rv ? (float)ei : -INFINITY;
        const float rs = rv ? pow2i(ei) : 0.f;
        const float rinv = rv ? pow2i(-ei) : 0.f;
        wait(kBarSFull, ph_s);
        tc::tc_fence_after();
        // S of this thread's row and head half (TMEM -> registers)
        auto load_s = [&](float (&v)[NH]) {
          if constexpr (NH % 32 == 0) {
#pragma unroll
            for (int g32 = 0; g32 < NH / 32; ++g32) {
              const uint32_t c = tl_lane + Cfg::kColS + half * NH + 32 * g32;
              uint32_t a[16], b[16];
              tc::tmem_ld16x2(c, c + 16, a, b);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                v[32 * g32 + i] = __uint_as_float(a[i]);
                v[32 * g32 + 16 + i] = __uint_as_float(b[i]);
              }
            }
          } else {
            tc::tmem_ld<NH>(tl_lane + Cfg::kColS + half * NH, v);
          }
        };
        // P as f16, MN-major [128 rows, HPG]
        auto store_p = [&](const float (&v)[NH]) {
#pragma unroll
          for (int k = 0; k < NH / 8; ++k) {
            uint32_t pw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pw[e] = tc::pack_f16x2(v[8 * k + 2 * e], v[8 * k + 2 * e + 1]);
            const int ci = half * (NH / 8) + k;
            const uint32_t po = p_off<HPG>(prow, ci);
            if (dbg_ok(p.status, po + 16u <= Cfg::kPBytes, kDbgSmemP))
              tc::st_shared_v4(p_base + po, pw[0], pw[1], pw[2], pw[3]);
          }
        };
        float x[NH];
        load_s(x);
        // Scores and, against the current running max, P -- optimistically:
        // the max moves on only when a score passes it by kRescaleSlack (a few
        // tiles per token), and then the whole group redoes P below.
        // (The token's first tile always raises the max from its initial
        // value: it goes straight to the exact pass.)
        bool need = first_pv;
        if (!first_pv) {
#pragma unroll
          for (int g4 = 0; g4 < NH / 4; ++g4) {
            const float4 m4 = m_s4[g4], f4 = hf_s4[g4];
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w}, hf[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float &xv = x[4 * g4 + i];
              const float t = fmaf(xv, hf[i] * rs, er - mm[i]);   // y - m (-inf if not kept)
              need |= t > kRescaleSlack;
              xv = tc::ex2(t);
            }
          }
          store_p(x);
          tc::fence_async_smem();
        }
        tc::tc_fence_before();
        if (sm_bar_or(need ? 1 : 0)) {
          // Raise the running max to the tile max; rescale sums and O; redo P.
          tc::tc_fence_after();
          load_s(x);
#pragma unroll
          for (int j = 0; j < NH; ++j) x[j] = fmaf(x[j], headf_s[half * NH + j] * rs, er);   // y
          // Per-head max over the warp's 32 rows by recursive halving, in
          // place (x is reloaded below): at step st a lane keeps the upper
          // half of its 2 st values when lane bit st is set, else the lower,
          // and takes the max with the partner's copy of that half; head j
          // ends in lane j (NH < 32: lanes j, j + NH, ... are folded last).
#pragma unroll
          for (int st = NH / 2; st >= 1; st >>= 1) {
            const bool up = (lane & st) != 0;
#pragma unroll
            for (int i = 0; i < st; ++i) {
              const float send = up ? x[i] : x[i + st];
              const float keep = up ? x[i + st] : x[i];
              x[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, st));
            }
          }
#pragma unroll
          for (int off = NH; off < 32; off <<= 1) x[0] = fmaxf(x[0], __shfl_xor_sync(0xffffffffu, x[0], off));
          if (lane < NH) red_s[q4 * 64 + half * NH + lane] = x[0];
          sm_bar();
          if (tid < HPG) {   // new max and rescale factor of head tid (factor -> red_s[tid])
            const float tm = fmaxf(fmaxf(red_s[tid], red_s[64 + tid]), fmaxf(red_s[128 + tid], red_s[192 + tid]));
            const float mo = m_s[tid];
            const float mn = fmaxf(mo, tm);
            red_s[tid] = tc::ex2(mo - mn);   // 0 when mo is still kMaxInit
            m_s[tid] = mn;
          }
          sm_bar();
#pragma unroll
          for (int j = 0; j < NH; ++j) l_reg[j] *= red_s[half * NH + j];
          if (!first_pv) {
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
              for (int g8 = 0; g8 < NH / 8; ++g8) {
                float o[8];
                const uint32_t ta = tl_lane + Cfg::kColO + mb * HPG + half * NH + 8 * g8;
                tc::tmem_ld<8>(ta, o);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] *= red_s[half * NH + 8 * g8 + i];
                tc::tmem_st<8>(ta, o);
              }
            }
          }
          load_s(x);
#pragma unroll
          for (int j = 0; j < NH; ++j) x[j] = fmaf(x[j], headf_s[half * NH + j] * rs, er);   // y
#pragma unroll
          for (int g4 = 0; g4 < NH / 4; ++g4) {
            const float4 m4 = m_s4[g4];
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float &xv = x[4 * g4 + i];
              xv = tc::ex2(xv - mm[i]);   // y = -inf (row not kept): 0
            }
          }
          store_p(x);
          tc::fence_async_smem();
          tc::tc_fence_before();
          sm_bar();   // P, O and red_s settled before PV
        }
#pragma unroll
        for (int j = 0; j < NH; ++j) l_reg[j] = fmaf(x[j], rinv, l_reg[j]);   // += 2^(x - m)
        // ---- O^T += K^T . P
        if (issuer && !*abort_s) {
          tc::tc_fence_after();
          // M blocks unrolled with compile-time indices (runtime-indexed
          // operands slowed the issue loop measurably).
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
            const uint64_t ab = dA_pv + (uint64_t)((2 * mb * 16384) >> 4);
            const uint32_t dt = tmem + Cfg::kColO + mb * HPG;
            tc::mma_f16(dt, ab, dB_pv, Cfg::kIdPV, first_pv ? 0u : 1u);
#pragma unroll
            for (int ks = 1; ks < 8; ++ks)
              tc::mma_f16(dt, ab + (uint64_t)((ks * 2048) >> 4),
                          dB_pv + (uint64_t)((ks * 16 * Cfg::kPRow) >> 4), Cfg::kIdPV, 1u);
            tc::mma_commit(&bars[kBarKvFree + mb]);
          }
          Cursor cv = cu;
          cursor_next_live(p, cv, seg.u_end);
          if (cv.u >= seg.u_end) tc::mma_commit(&bars[kBarOFinal]);   // last PV of this token
        }
        __syncwarp();
        first_pv = false;
      }
      finalize(seg);
    }
  }

  // After a wait gave up, MMAs issued before it may still be running: the
  // issuer commits once more and waits (with the full default budget, MMAs
  // always finish) until every one of them is done, so TMEM is never freed
  // under a running MMA.
  if (tid == 0 && *abort_s) {
    tc::mma_commit(&bars[kBarDrain]);
    tc::mbar_wait(&bars[kBarDrain], 0u, kWaitBudget);
  }
  if constexpr (kPQ) {   // the producers' lane 0 threads likewise (each may have issued QKs)
    if (warp >= kSmWarps && lane == 0 && *abort_s) {
      tc::mma_commit(&bars[kBarDrainQK]);
      tc::mbar_wait(&bars[kBarDrainQK], 0u, kWaitBudget);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cfg::kCols);
  }
}

}  // namespace dsa

bool dsa_tc_supports(int hpg) { return hpg == 16 || hpg == 32 || hpg == 64; }

namespace {
// Checks that the kernel kept exactly kLaunchRegs registers per thread (the
// warpgroup register split assumes it) and raises its shared-memory limit.
template <int N, bool E, bool S, bool M, bool V = false, bool SH = false, bool PQ = false>
cudaError_t tc_setup(void *) {
  using namespace dsa;
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, tc_decode_kernel<N, E, S, M, V, SH, PQ>);
  if (err != cudaSuccess) return err;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(tc_decode_kernel<N, E, S, M, V, SH, PQ>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)TcCfg<N, V>::kSmem);
}

// V3.2 records (576-dim keys): groups of 16 or 32 heads only.
template <int N>
cudaError_t launch_v32(const dsa::Params &p, dim3 grid, dim3 block, cudaStream_t stream, int bit) {
  using namespace dsa;
  if constexpr (N > 32) {
    return cudaErrorInvalidValue;
  } else {
    const cudaError_t err = dsa_configure_once(bit, &tc_setup<N, false, false, false, true>, nullptr);
    if (err != cudaSuccess) return err;
    tc_decode_kernel<N, false, false, false, true>
        <<<grid, block, (int)TcCfg<N, true>::kSmem, stream>>>(p);
    return cudaSuccess;
  }
}

// The plain form: head groups sharing tiles or not (SH), and at 64 heads per
// group with `pq` the form whose producers stage Q (kPQ).
template <int N, bool SH>
cudaError_t launch_plain(const dsa::Params &p, bool pq, dim3 grid, dim3 block,
                         cudaStream_t stream, int bit, int bit_pq) {
  using namespace dsa;
  const int smem = (int)TcCfg<N>::kSmem;
  if constexpr (N == 64) {
    if (pq) {
      const cudaError_t err =
          dsa_configure_once(bit_pq, &tc_setup<N, false, false, false, false, SH, true>, nullptr);
      if (err != cudaSuccess) return err;
      tc_decode_kernel<N, false, false, false, false, SH, true><<<grid, block, smem, stream>>>(p);
      return cudaSuccess;
    }
  }
  const cudaError_t err =
      dsa_configure_once(bit, &tc_setup<N, false, false, false, false, SH>, nullptr);
  if (err != cudaSuccess) return err;
  tc_decode_kernel<N, false, false, false, false, SH><<<grid, block, smem, stream>>>(p);
  return cudaSuccess;
}
}  // namespace

cudaError_t dsa_launch_tc(const dsa::Params &p, cudaStream_t stream) {
  using namespace dsa;
  const dim3 grid((unsigned)(p.C * p.HG)), block(kTcThreads);
  auto has_fmt = [&](int32_t f) {
    return p.list[0].fmt == f || (p.nlists > 1 && p.list[1].fmt == f);
  };
  const bool m1 = has_fmt(DSA_REC_MODEL1_584);
  const bool v32 = p.dqk == 576;
  const bool ext = p.rope_gptj || p.mx_on || has_fmt(DSA_REC_FP8_528_UE8M0);
  // exact-budget waits (a plan with a wait budget) exist for the plain form
  const bool strict = !ext && p.wait_budget > 0;
  // the plan's choice of the form whose producers stage Q (kPQ)
  const bool pq = p.pq != 0;
  cudaError_t err = cudaSuccess;
  switch (p.hpg) {
#define DSA_TC_CASE(N, BIT)                                                                   \
  case N: {                                                                                   \
    const int smem = (int)TcCfg<N>::kSmem;                                                    \
    if (v32) {                                                                                \
      err = launch_v32<N>(p, grid, block, stream, BIT + 36);                                  \
      if (err != cudaSuccess) return err;                                                     \
    } else if (m1 && ext) {                                                                   \
      err = dsa_configure_once(BIT + 28, &tc_setup<N, true, false, true>, nullptr);           \
      if (err != cudaSuccess) return err;                                                     \
      tc_decode_kernel<N, true, false, true, false><<<grid, block, smem, stream>>>(p);        \
    } else if (m1) {                                                                          \
      err = dsa_configure_once(BIT + 32, &tc_setup<N, false, false, true>, nullptr);          \
      if (err != cudaSuccess) return err;                                                     \
      tc_decode_kernel<N, false, false, true, false><<<grid, block, smem, stream>>>(p);       \
    } else if (ext) {                                                                         \
      err = dsa_configure_once(BIT + 20, &tc_setup<N, true, false, false>, nullptr);          \
      if (err != cudaSuccess) return err;                                                     \
      tc_decode_kernel<N, true, false, false, false><<<grid, block, smem, stream>>>(p);       \
    } else if (strict) {                                                                      \
      err = dsa_configure_once(BIT + 24, &tc_setup<N, false, true, false>, nullptr);          \
      if (err != cudaSuccess) return err;                                                     \
      tc_decode_kernel<N, false, true, false, false><<<grid, block, smem, stream>>>(p);       \
    } else if (p.HG > 1) {                                                                    \
      err = launch_plain<N, true>(p, pq, grid, block, stream, BIT + 40, BIT + 44);            \
      if (err != cudaSuccess) return err;                                                     \
    } else {                                                                                  \
      err = launch_plain<N, false>(p, pq, grid, block, stream, BIT, BIT + 48);                \
      if (err != cudaSuccess) return err;                                                     \
    }                                                                                         \
    break;                                                                                    \
  }
    DSA_TC_CASE(16, 0)
    DSA_TC_CASE(32, 1)
    DSA_TC_CASE(64, 2)
#undef DSA_TC_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
