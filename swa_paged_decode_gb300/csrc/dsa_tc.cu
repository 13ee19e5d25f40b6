// dsa_tc.cu -- fused gather + dequant + attention on sm_103a tensor cores.
//
// One persistent CTA (256 threads, one per SM: its shared memory forbids a
// second) walks a contiguous range of (token, 128-row tile) units. Per tile:
//
//   gather   predicated 16-byte loads of the tile's 128 records (2 threads
//            per row), issued one tile ahead so they are in flight while the
//            previous tile computes;
//   dequant  records -> f16 K-major tile in shared memory, 128-byte swizzle
//            (16-byte chunk c of row r stored at chunk c ^ (r % 8));
//            NVFP4: e2m1 * e4m3 scale (exact in f16);
//            fp8:   e4m3 * s_hi, where s_hi is the fp32 block scale rounded to
//            7 significant bits (product exact in f16); the remaining factor
//            rho = s / s_hi (fp32, per row and 128-dim block) is applied to
//            the block scores and, for PV, to P of the matching 128-dim M
//            block, so both products see the exact dequantized row;
//   QK^T     swap-AB: S[128 rows, H] = K[128, 512] . Q[H, 512]^T with
//            tcgen05.mma kind::f16 into TMEM (fp8 tiles: one accumulator per
//            128-dim scale block, scaled by rho in fp32 afterwards);
//   softmax  one TMEM lane (= one KV row) per thread pair, base-2, with a
//            running per-head max that is only raised when a score exceeds
//            it by more than 2^8 (then O in TMEM and the partial sums are
//            rescaled) -- the common tile needs no cross-row max at all;
//   PV       O^T[512, H] += K^T[512, 128] . P[128, H], four 128-dim M blocks,
//            A read MN-major from the same shared tile, accumulated in TMEM.
//
// At the end of a token: per-head sums reduced over rows, sink folded into
// the denominator, bf16 out and fp32 lse written (or an fp32 partial for a
// token split over CTAs, merged later by the combine kernel).
//
// Design sources (prior art, re-derived for this GPU): the vLLM
// "swapab_decode_attn" page (SwapABDecodeKernel: swap-AB tcgen05 tiles of 128
// KV rows, K-major SW128 KV tile read MN-major for PV, predicated 16-byte
// record loads, base-2 softmax), FlashMLA's sparse_decode.h page (split-KV
// partials + combine).
#include "dsa_internal.cuh"
#include "tc_ptx.cuh"

namespace dsa {

constexpr int kTcThreads = 256;
constexpr long long kWaitIters = 4000000000ll;  // wait budget in SM cycles (~2 s)
constexpr float kRescaleSlack = 8.0f;       // log2 headroom before the running max moves

template <int HPG>
struct TcCfg {
  static constexpr int kHalf = HPG / 2;                  // heads per thread
  static constexpr int kPRow = HPG * 2;                  // bytes per P row
  static constexpr int kPBufs = HPG == 64 ? 2 : 4;       // P' buffers (fp8 tiles: one per M block)
  static constexpr uint32_t kPBytes = 128 * kPRow;       // one P tile
  static constexpr uint32_t kKV = 0;                     // 128 x 512 f16 = 128 KiB
  static constexpr uint32_t kQ = 131072;                 // HPG x 512 f16
  static constexpr uint32_t kP = kQ + HPG * 1024;        // kPBufs x [128 x HPG] f16
  static constexpr uint32_t kHeadF = kP + kPBufs * kPBytes;  // [64] f32 per-head score factor
  static constexpr uint32_t kM = kHeadF + 256;           // [64] running max (log2)
  static constexpr uint32_t kAlpha = kM + 256;           // [64]
  static constexpr uint32_t kInv = kAlpha + 256;         // [64]
  static constexpr uint32_t kRed = kInv + 256;           // [4][64] f32
  static constexpr uint32_t kMisc = kRed + 1024;         // flags, mbarriers, tmem base
  static constexpr uint32_t kBytes = kMisc + 64;
  // Dynamic shared memory requested: the tiles plus slack for aligning the
  // base to 1024 bytes, capped at the 227 KiB a CTA may use.
  static constexpr uint32_t kSmem = kBytes + 1024 > 232448u ? 232448u : kBytes + 1024;
  static constexpr uint32_t kCols = HPG == 16 ? 128 : (HPG == 32 ? 256 : 512);
  static constexpr uint32_t kColS = 0;                   // S block b at b*HPG
  static constexpr uint32_t kColO = 4 * HPG;             // O block mb at (4+mb)*HPG
  static constexpr uint32_t kPSwz = HPG == 64 ? tc::kSwz128 : (HPG == 32 ? tc::kSwz64 : tc::kSwz32);
  static constexpr uint32_t kIdQK = tc::idesc_f16(128, HPG, false, false);
  static constexpr uint32_t kIdPV = tc::idesc_f16(128, HPG, true, true);
  static_assert(kBytes <= 232448u, "shared memory layout exceeds 227 KiB");
};

// Byte offset of the 16-byte chunk holding f16 elements [8*ci, 8*ci+8) of
// row r in a K-major 128B-swizzled tile whose k-blocks are `kb_bytes` apart.
__device__ __forceinline__ uint32_t sw128_off(int r, int kb, int ci, uint32_t kb_bytes) {
  return (uint32_t)kb * kb_bytes + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
         (uint32_t)((ci ^ (r & 7)) << 4);
}

// P tile (MN-major: row r holds HPG f16 heads), swizzle matching its row width.
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

// Per-thread prefetch registers for one tile. Thread (warp w, lane l) owns
// row 32*(w%4) + l -- the TMEM lane its softmax reads -- and half j = w/4 of
// the record's 16-byte chunks: c = 4m + 2j + e (e in {0,1}), i.e. whole
// 32-byte sectors.
struct Gather {
  uint4 d[16];   // fp8: 16 chunks; NVFP4: 8 chunks
  uint4 s[2];    // fp8: s[0] = 4 fp32 scales; NVFP4: 32 e4m3 scales
  int32_t sid;
  int32_t r;
  bool ok;
};

__device__ __forceinline__ void unit_info(const Params &p, int64_t u, int32_t &t, int32_t &lid,
                                          int32_t &row0) {
  t = (int32_t)(u / p.tpt);
  unit_tile(p, u, lid, row0);
}

__device__ __forceinline__ void prefetch(const Params &p, int64_t u, Gather &g) {
  int32_t t, lid, row0;
  unit_info(p, u, t, lid, row0);
  const ListArgs &L = p.list[lid];
  const int row = 32 * ((threadIdx.x >> 5) & 3) + (threadIdx.x & 31), j = threadIdx.x >> 7;
  g.r = row0 + row;
  g.sid = -1;
  if (g.r < L.width) g.sid = __ldg(L.ids + (int64_t)t * L.idx_stride + g.r);
  const int32_t limit = list_limit(L, t);
  g.ok = slot_valid(L, g.r, limit, g.sid);
  const uint4 z = make_uint4(0, 0, 0, 0);
  if (L.fmt == DSA_REC_FP8_528) {
    if (g.ok) {
      const uint8_t *rec = record_ptr(L, g.sid);
#pragma unroll
      for (int k = 0; k < 16; ++k) g.d[k] = tc::ldg_nc_v4(rec + 16 * (4 * (k >> 1) + 2 * j + (k & 1)));
      g.s[0] = tc::ldg_nc_v4(rec + 512);
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) g.d[k] = z;
      g.s[0] = z;
    }
  } else {
    if (g.ok) {
      const uint8_t *rec = record_ptr(L, g.sid);
#pragma unroll
      for (int k = 0; k < 8; ++k) g.d[k] = tc::ldg_nc_v4(rec + 16 * (4 * (k >> 1) + 2 * j + (k & 1)));
      g.s[0] = tc::ldg_nc_v4(rec + 256);
      g.s[1] = tc::ldg_nc_v4(rec + 272);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) g.d[k] = z;
      g.s[0] = z;
      g.s[1] = z;
    }
  }
}

// fp32 block scale -> (f16 s_hi with 7 significant bits, rho = s / s_hi).
__device__ __forceinline__ void split_scale(float s, uint32_t &shi2, float &rho) {
  uint32_t u = __float_as_uint(s);
  u = (u + 0x10000u) & 0xFFFE0000u;        // round to 6 explicit mantissa bits
  const __half h = __float2half_rn(__uint_as_float(u));
  const float hf = __half2float(h);
  rho = (hf != 0.f) ? s / hf : 0.f;
  const uint32_t hb = (uint32_t)__half_as_ushort(h);
  shi2 = hb | (hb << 16);
}

// Registers -> f16 tile in shared memory. fp8 records also return the four
// per-block factors rho = s / s_hi of this thread's row.
__device__ __forceinline__ void dequant(const Params &p, int32_t lid, const Gather &g,
                                        uint32_t kv_base, float (&rho)[4]) {
  const ListArgs &L = p.list[lid];
  const int row = 32 * ((threadIdx.x >> 5) & 3) + (threadIdx.x & 31), j = threadIdx.x >> 7;
  if (L.fmt == DSA_REC_FP8_528) {
    uint32_t shi2[4];
    split_scale(__uint_as_float(g.s[0].x), shi2[0], rho[0]);
    split_scale(__uint_as_float(g.s[0].y), shi2[1], rho[1]);
    split_scale(__uint_as_float(g.s[0].z), shi2[2], rho[2]);
    split_scale(__uint_as_float(g.s[0].w), shi2[3], rho[3]);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int c = 4 * (k >> 1) + 2 * j + (k & 1);  // dims [16c, 16c+16), scale block c/8
      const uint32_t sc = shi2[c >> 3];
      const uint32_t w[4] = {g.d[k].x, g.d[k].y, g.d[k].z, g.d[k].w};
      uint32_t f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        tc::e4m3x4_to_f16x4(w[i], f[2 * i], f[2 * i + 1]);
        f[2 * i] = tc::hmul2(f[2 * i], sc);
        f[2 * i + 1] = tc::hmul2(f[2 * i + 1], sc);
      }
      const int kb = c >> 2, ci = (2 * c) & 7;
      tc::st_shared_v4(kv_base + sw128_off(row, kb, ci, 16384), f[0], f[1], f[2], f[3]);
      tc::st_shared_v4(kv_base + sw128_off(row, kb, ci + 1, 16384), f[4], f[5], f[6], f[7]);
    }
  } else {
    rho[0] = rho[1] = rho[2] = rho[3] = 1.f;
    const uint32_t sw[8] = {g.s[0].x, g.s[0].y, g.s[0].z, g.s[0].w,
                            g.s[1].x, g.s[1].y, g.s[1].z, g.s[1].w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = 4 * (k >> 1) + 2 * j + (k & 1);  // dims [32c, 32c+32), scales 2c, 2c+1
      const uint32_t pair = (sw[c >> 1] >> (16 * (c & 1))) & 0xFFFFu;
      const uint32_t s2 = tc::e4m3x2_to_f16x2(pair);
      const uint32_t sa = __byte_perm(s2, s2, 0x1010), sb = __byte_perm(s2, s2, 0x3232);
      const uint32_t w[4] = {g.d[k].x, g.d[k].y, g.d[k].z, g.d[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // word i = dims [32c + 8i, 32c + 8i + 8)
        uint32_t f[4];
        tc::e2m1x8_to_f16x8(w[i], f);
        const uint32_t sc = i < 2 ? sa : sb;
#pragma unroll
        for (int e = 0; e < 4; ++e) f[e] = tc::hmul2(f[e], sc);
        const int kb = c >> 1, ci = (4 * c + i) & 7;
        tc::st_shared_v4(kv_base + sw128_off(row, kb, ci, 16384), f[0], f[1], f[2], f[3]);
      }
    }
  }
}

template <int HPG>
__global__ void __launch_bounds__(kTcThreads, 1) tc_decode_kernel(Params p) {
  using Cfg = TcCfg<HPG>;
  constexpr int NH = Cfg::kHalf;
  extern __shared__ uint8_t smem_raw[];
  // Swizzled tiles need a 1024-byte aligned base (the swizzle acts on
  // address bits); the layout is checked to fit after aligning.
  const uint32_t raw_base = tc::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  if (pad + Cfg::kBytes > Cfg::kSmem) {
    if (threadIdx.x == 0) report_status(p.status, DSA_ERR_UNSUPPORTED);
    return;
  }
  uint8_t *smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;
  const uint32_t kv_base = sbase + Cfg::kKV;
  const uint32_t q_base = sbase + Cfg::kQ;
  const uint32_t p_base = sbase + Cfg::kP;
  float *headf_s = reinterpret_cast<float *>(smem + Cfg::kHeadF);
  float *m_s = reinterpret_cast<float *>(smem + Cfg::kM);
  float *alpha_s = reinterpret_cast<float *>(smem + Cfg::kAlpha);
  float *inv_s = reinterpret_cast<float *>(smem + Cfg::kInv);
  float *red_s = reinterpret_cast<float *>(smem + Cfg::kRed);
  int32_t *flag_s = reinterpret_cast<int32_t *>(smem + Cfg::kMisc);
  int32_t *err_s = flag_s + 1;
  uint32_t *red_u = reinterpret_cast<uint32_t *>(flag_s + 2);   // [2] selection reduction
  uint64_t *bar_s = reinterpret_cast<uint64_t *>(smem + Cfg::kMisc + 16);
  uint64_t *bar_o = bar_s + 1;
  uint64_t *bar_p = bar_s + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kMisc + 48);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, half = warp >> 2;
  const int prow = 32 * q4 + lane;   // TMEM lane = KV row handled in the softmax
  const int hg = blockIdx.x % p.HG;
  const int cta = blockIdx.x / p.HG;
  const int h0 = hg * HPG;
  const int64_t u0 = cta_unit_begin(p, cta), u1 = cta_unit_end(p, cta);
  if (u0 >= u1) return;

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, Cfg::kCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar_s, 1);
    tc::mbar_init(bar_o, 1);
    tc::mbar_init(bar_p, 1);
    tc::fence_mbar_init();
    *flag_s = 0;
    *err_s = 0;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl_lane = tmem + ((uint32_t)(32 * q4) << 16);   // this warp's TMEM lanes

  uint32_t ph_s = 0, ph_o = 0, ph_p = 0;
  bool o_pending = false;
  bool failed = false;
  float m_reg[NH], l_reg[NH];
  bool first_pv = true;
  uint32_t kept = 0, chk = 0;
  Segment seg;
  seg.t = -1;

  Gather g;
  prefetch(p, u0, g);

  // Wait for the last PV (O and the shared tiles are free afterwards).
  auto wait_o = [&]() {
    if (o_pending) {
      if (!tc::mbar_wait(bar_o, ph_o, kWaitIters)) failed = true;
      ph_o ^= 1;
      o_pending = false;
      tc::tc_fence_after();
    }
  };

  // Returns false (CTA-uniformly) when a bounded wait gave up.
  auto finalize = [&]() -> bool {
    wait_o();
    // Row selection record.
    uint32_t k2 = kept, c2 = chk;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      k2 += __shfl_xor_sync(0xffffffffu, k2, off);
      c2 += __shfl_xor_sync(0xffffffffu, c2, off);
    }
    // Per-head sums over rows: butterfly within the warp, then 4 quadrants.
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      float v = l_reg[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) red_s[q4 * 64 + half * NH + j] = v;
    }
    if (tid == 0) {
      red_u[0] = 0;
      red_u[1] = 0;
    }
    if (__syncthreads_or(failed ? 1 : 0)) {
      failed = true;
      return false;
    }
    if (lane == 0) {
      atomicAdd(&red_u[0], k2);
      atomicAdd(&red_u[1], c2);
    }
    if (tid < HPG) {
      const int h = tid;
      const float l = red_s[h] + red_s[64 + h] + red_s[128 + h] + red_s[192 + h];
      const float m = m_s[h];
      const float lse = (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
      float inv = 0.f;
      if (l > 0.f) {
        float den = l;
        if (seg.whole && p.sink) {
          const float sk = __ldg(p.sink + h0 + h);
          den = (sk == INFINITY) ? INFINITY : l + tc::ex2(sk * kLog2e - m);
        }
        inv = 1.f / den;
      }
      inv_s[h] = inv;
      if (seg.whole)
        p.lse[(int64_t)seg.t * p.H + h0 + h] = lse;
      else
        p.part_lse[((int64_t)hg * 2 * p.C + seg.slot) * HPG + h] = lse;
    }
    __syncthreads();
    if (hg == 0 && tid == 0) {
      int32_t *dst = seg.whole ? (p.sel + 2 * (int64_t)seg.t) : (p.part_sel + 2 * (int64_t)seg.slot);
      dst[0] = (int32_t)red_u[0];
      dst[1] = (int32_t)red_u[1];
    }
    // O^T[d, h] from TMEM: thread holds d = 128*mb + prow for its NH heads.
#pragma unroll 1
    for (int mb = 0; mb < 4; ++mb) {
      float o[NH];
      if (!first_pv) {
        tc::tmem_ld<NH>(tl_lane + Cfg::kColO + mb * HPG + half * NH, o);
      }
      const int d = 128 * mb + prow;
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const int h = half * NH + j;
        const float inv = inv_s[h];
        const float v = (first_pv || inv == 0.f) ? 0.f : o[j] * inv;
        if (seg.whole)
          p.out[((int64_t)seg.t * p.H + h0 + h) * kD + d] = __float2bfloat16_rn(v);
        else
          p.part_o[(((int64_t)hg * 2 * p.C + seg.slot) * HPG + h) * kD + d] = v;
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    return true;
  };

  auto stage_q = [&](int32_t t) {
    int64_t pos = p.positions ? __ldg(p.positions + t) : 0;
    if (pos < 0 || (p.cos_sin && pos >= p.cs_rows)) {   // outside the table: flag, use row 0
      if (tid == 0) report_status(p.status, DSA_ERR_INVALID_ARG);
      pos = 0;
    }
    for (int h = warp; h < HPG; h += kTcThreads / 32) {
      const __nv_bfloat16 *qh = p.q + (int64_t)t * p.q_st + (int64_t)(h0 + h) * p.q_sh;
      const uint4 a = __ldg(reinterpret_cast<const uint4 *>(qh) + 2 * lane);
      const uint4 b = __ldg(reinterpret_cast<const uint4 *>(qh) + 2 * lane + 1);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
      }
      if (p.cos_sin) {   // NeoX: dim 448+i pairs with 480+i; lanes 28..31 hold 448..511
        const float *cs = p.cos_sin + pos * 64;
        const bool rope = lane >= 28;
        const bool first = lane < 30;
        const int i0 = (lane & 1) * 16;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float other = __shfl_xor_sync(0xffffffffu, v[k], 2);
          if (rope) {
            const float c = __ldg(cs + i0 + k), s = __ldg(cs + kRopeHalf + i0 + k);
            v[k] = first ? (v[k] * c - other * s) : (v[k] * c + other * s);
          }
        }
      }
      float mx = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) mx = fmaxf(mx, fabsf(v[k]));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      int e = (mx > 0.f) ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
      e = e < -126 ? -126 : (e > 126 ? 126 : e);
      const float down = __uint_as_float((uint32_t)(127 - e) << 23);
      const float up = __uint_as_float((uint32_t)(127 + e) << 23);
      if (lane == 0) headf_s[h] = p.scale_log2 * up;
      uint32_t f[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = tc::pack_f16x2(v[2 * i] * down, v[2 * i + 1] * down);
      const int kb = lane >> 2, ci = (lane & 3) * 2;
      tc::st_shared_v4(q_base + sw128_off(h, kb, ci, HPG * 128), f[0], f[1], f[2], f[3]);
      tc::st_shared_v4(q_base + sw128_off(h, kb, ci + 1, HPG * 128), f[4], f[5], f[6], f[7]);
    }
    if (tid < HPG) m_s[tid] = -INFINITY;
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      m_reg[j] = -INFINITY;
      l_reg[j] = 0.f;
    }
    first_pv = true;
    kept = 0;
    chk = 0;
  };

  for (int64_t u = u0; u < u1 && !failed; ++u) {
    int32_t t, lid, row0;
    unit_info(p, u, t, lid, row0);
    if (t != seg.t) {
      if (seg.t >= 0 && !finalize()) break;
      seg = make_segment(p, cta, t);
      stage_q(t);
    }
    wait_o();
    const bool fp8 = p.list[lid].fmt == DSA_REC_FP8_528;
    float rho[4];
    dequant(p, lid, g, kv_base, rho);
    const bool row_ok = g.ok;
    if (half == 0 && g.ok) {
      kept += 1;
      chk += row_hash(g.sid, g.r, lid);
    }
    tc::fence_async_smem();
    tc::tc_fence_before();
    const int st = __syncthreads_or((row_ok ? 1 : 0) | (failed ? 2 : 0));
    tc::tc_fence_after();
    if (st & 2) {
      failed = true;
      break;
    }
    if (u + 1 < u1) prefetch(p, u + 1, g);
    if (!(st & 1)) continue;

    // ---- S = K . Q^T
    if (tid == 0) {
#pragma unroll 1
      for (int kb = 0; kb < 8; ++kb) {
        const uint32_t d_tmem = tmem + Cfg::kColS + (fp8 ? (uint32_t)(kb >> 1) * HPG : 0u);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = tc::sdesc(kv_base + kb * 16384 + ks * 32, 16, 1024, tc::kSwz128);
          const uint64_t bd = tc::sdesc(q_base + kb * HPG * 128 + ks * 32, 16, 1024, tc::kSwz128);
          const uint32_t acc = fp8 ? ((kb & 1) | ks) : (kb | ks);
          tc::mma_f16(d_tmem, ad, bd, Cfg::kIdQK, acc);
        }
      }
      tc::mma_commit(bar_s);
    }
    const bool s_late = !tc::mbar_wait(bar_s, ph_s, kWaitIters);
    ph_s ^= 1;
    tc::tc_fence_after();

    // ---- softmax on this thread's row and NH heads
    float x[NH];
    {
      const bool rv = row_ok;
      if (fp8) {
#pragma unroll
        for (int j = 0; j < NH; ++j) x[j] = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float sv[NH];
          tc::tmem_ld<NH>(tl_lane + Cfg::kColS + b * HPG + half * NH, sv);
#pragma unroll
          for (int j = 0; j < NH; ++j) x[j] = fmaf(rho[b], sv[j], x[j]);
        }
      } else {
        tc::tmem_ld<NH>(tl_lane + Cfg::kColS + half * NH, x);
      }
      bool need = false;
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        x[j] = rv ? x[j] * headf_s[half * NH + j] : -INFINITY;
        need |= x[j] > m_reg[j] + kRescaleSlack;
      }
      if (__any_sync(0xffffffffu, need) && lane == 0) *flag_s = 1;
    }
    if (__syncthreads_or(s_late ? 1 : 0)) {
      failed = true;
      break;
    }
    if (*flag_s) {
      // Raise the running max to the tile max; rescale partial sums and O.
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        float v = x[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) red_s[q4 * 64 + half * NH + j] = v;
      }
      __syncthreads();
      if (tid < HPG) {
        const float tm = fmaxf(fmaxf(red_s[tid], red_s[64 + tid]), fmaxf(red_s[128 + tid], red_s[192 + tid]));
        const float mo = m_s[tid];
        const float mn = fmaxf(mo, tm);
        alpha_s[tid] = (mn == -INFINITY) ? 1.f : (mo == -INFINITY ? 0.f : tc::ex2(mo - mn));
        m_s[tid] = mn;
      }
      __syncthreads();
      float al[NH];
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        al[j] = alpha_s[half * NH + j];
        m_reg[j] = m_s[half * NH + j];
        l_reg[j] *= al[j];
      }
      if (!first_pv) {
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
          float o[NH];
          const uint32_t ta = tl_lane + Cfg::kColO + mb * HPG + half * NH;
          tc::tmem_ld<NH>(ta, o);
#pragma unroll
          for (int j = 0; j < NH; ++j) o[j] *= al[j];
          tc::tmem_st<NH>(ta, o);
        }
      }
    }
    // P = 2^(x - m) (<= 2^8); f16, MN-major [128 rows, HPG].
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      x[j] = (x[j] == -INFINITY) ? 0.f : tc::ex2(x[j] - m_reg[j]);
      l_reg[j] += x[j];
    }
    // NVFP4 tiles: one P for all four M blocks. fp8 tiles: P'_mb = P * rho_mb
    // for M block mb, written kPBufs at a time.
    const int nbatch = fp8 ? 4 / Cfg::kPBufs : 1;
    bool late = false;
    for (int batch = 0; batch < nbatch; ++batch) {
      if (batch > 0) {   // the previous batch's MMAs must be done reading P'
        late |= !tc::mbar_wait(bar_p, ph_p, kWaitIters);
        ph_p ^= 1;
        tc::tc_fence_after();
      }
      const int nb = fp8 ? Cfg::kPBufs : 1;
      for (int i = 0; i < nb; ++i) {
        const float f = fp8 ? rho[batch * nb + i] : 1.f;
        uint32_t pw[NH / 2];
#pragma unroll
        for (int j = 0; j < NH; j += 2) pw[j / 2] = tc::pack_f16x2(x[j] * f, x[j + 1] * f);
#pragma unroll
        for (int k = 0; k < NH / 8; ++k) {
          const int ci = half * (NH / 8) + k;
          tc::st_shared_v4(p_base + i * Cfg::kPBytes + p_off<HPG>(prow, ci), pw[4 * k],
                           pw[4 * k + 1], pw[4 * k + 2], pw[4 * k + 3]);
        }
      }
      tc::fence_async_smem();
      tc::tc_fence_before();
      if (__syncthreads_or(late ? 1 : 0)) {
        failed = true;
        break;
      }
      // ---- O^T += K^T . P
      if (tid == 0) {
        *flag_s = 0;
        tc::tc_fence_after();
        const int mb0 = fp8 ? batch * Cfg::kPBufs : 0;
        const int mb1 = fp8 ? mb0 + Cfg::kPBufs : 4;
#pragma unroll 1
        for (int mb = mb0; mb < mb1; ++mb) {
          const uint32_t pb = p_base + (fp8 ? (uint32_t)(mb - mb0) * Cfg::kPBytes : 0u);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad =
                tc::sdesc(kv_base + 2 * mb * 16384 + ks * 2048, 16384, 1024, tc::kSwz128);
            const uint64_t bd = tc::sdesc(pb + ks * 16 * Cfg::kPRow, Cfg::kPBytes,
                                          8 * Cfg::kPRow, Cfg::kPSwz);
            tc::mma_f16(tmem + Cfg::kColO + mb * HPG, ad, bd, Cfg::kIdPV,
                        (first_pv && ks == 0) ? 0u : 1u);
          }
        }
        tc::mma_commit(batch + 1 < nbatch ? bar_p : bar_o);
      }
    }
    if (failed) break;
    o_pending = true;
    first_pv = false;
  }
  if (!failed && seg.t >= 0) finalize();
  if (failed) {
    report_status(p.status, DSA_ERR_TIMEOUT);
    // Give outstanding tensor-core work a bounded chance to drain.
    if (o_pending) tc::mbar_wait(bar_o, ph_o, kWaitIters);
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

cudaError_t dsa_launch_tc(const dsa::Params &p, cudaStream_t stream) {
  using namespace dsa;
  const dim3 grid((unsigned)(p.C * p.HG)), block(kTcThreads);
  cudaError_t err = cudaSuccess;
  switch (p.hpg) {
#define DSA_TC_CASE(N)                                                                   \
  case N: {                                                                              \
    const int smem = (int)TcCfg<N>::kSmem;                                               \
    err = cudaFuncSetAttribute(tc_decode_kernel<N>,                                      \
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);       \
    if (err != cudaSuccess) return err;                                                  \
    tc_decode_kernel<N><<<grid, block, smem, stream>>>(p);                               \
    break;                                                                               \
  }
    DSA_TC_CASE(16)
    DSA_TC_CASE(32)
    DSA_TC_CASE(64)
#undef DSA_TC_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
