// dsa_simt.cu -- correctness-first CUDA-core decode kernel.
//
// Same schedule, selection, record decoding and output contract as the
// tensor-core kernel; every product in fp32 FMAs. Used as a cross-check and
// for head counts the tensor-core kernel does not take.
//
// One CTA of 256 threads walks its contiguous (token, tile) range; a tile is
// processed as four 32-row sub-tiles: gather + dequantize to fp32 shared
// memory, scores, an online softmax in base 2 (running max per head), then
// the P.V update of the fp32 accumulator held in registers.
#include "dsa_internal.cuh"

namespace dsa {

constexpr int kSimtThreads = 256;
constexpr int kSub = 32;  // rows per sub-tile

struct SimtSmem {
  float q[64 * kD];        // Q rows of the head group (fp32, RoPE applied)
  float k[kSub * kD];      // dequantized rows of the sub-tile
  float s[64 * kSub];      // scores, then probabilities
  float m[64];             // running max (log2 units)
  float l[64];             // running sum
  float alpha[64];         // rescale factor of this sub-tile
  int32_t valid[kSub];
  int32_t red[2 * (kSimtThreads / 32)];
};

// Gather + dequantize rows [row0, row0+32) of list `lid` for token t into
// sm.k (invalid rows zero, sm.valid[i] = 0). 8 threads per row.
__device__ void load_subtile(const Params &p, SimtSmem &sm, int32_t lid, int32_t t,
                             int32_t row0, uint32_t &kept, uint32_t &chk) {
  const ListArgs &L = p.list[lid];
  const int tid = threadIdx.x;
  const int i = tid >> 3, j = tid & 7;
  const int32_t r = row0 + i;
  const int32_t limit = list_limit(L, t);
  int32_t sid = -1;
  if (r < L.width) sid = __ldg(L.ids + (int64_t)t * L.idx_stride + r);
  const bool ok = slot_valid(L, r, limit, sid);
  float *krow = sm.k + i * kD;
  if (!ok) {
    for (int d = j; d < kD; d += 8) krow[d] = 0.f;
  } else if (L.fmt == DSA_REC_MODEL1_584) {   // 8-byte aligned records: 8-byte loads
    const uint8_t *rec = record_ptr(L, sid);
    const uint2 sc = __ldg(reinterpret_cast<const uint2 *>(rec + 576));   // 7 ue8m0 + 1 unused
#pragma unroll
    for (int kk = 0; kk < 7; ++kk) {
      const int w = j + 8 * kk;   // 8-byte word = dims [8w, 8w+8), in 64-dim block kk
      const uint2 v = __ldg(reinterpret_cast<const uint2 *>(rec) + w);
      const float s = ue8m0_to_f32((kk < 4 ? sc.x : sc.y) >> (8 * (kk & 3)));
#pragma unroll
      for (int e = 0; e < 8; ++e)
        krow[8 * w + e] = e4m3_to_f32(((e < 4 ? v.x : v.y) >> (8 * (e & 3))) & 0xFFu) * s;
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int w = j + 8 * kk;   // bf16 dims 448 + [4w, 4w+4)
      const uint2 v = __ldg(reinterpret_cast<const uint2 *>(rec + 448) + w);
      krow[448 + 4 * w + 0] = bf16_bits_to_f32(v.x & 0xFFFFu);
      krow[448 + 4 * w + 1] = bf16_bits_to_f32(v.x >> 16);
      krow[448 + 4 * w + 2] = bf16_bits_to_f32(v.y & 0xFFFFu);
      krow[448 + 4 * w + 3] = bf16_bits_to_f32(v.y >> 16);
    }
  } else if (L.fmt != DSA_REC_NVFP4_288) {   // fp8: fp32 scales per 128 or ue8m0 per 32 dims
    const uint8_t *rec = record_ptr(L, sid);
    const bool ue = L.fmt == DSA_REC_FP8_528_UE8M0;
    const uint4 sc = __ldg(reinterpret_cast<const uint4 *>(rec + 512));
    const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int c = j + 8 * kk;  // 16-byte chunk = dims [16c, 16c+16)
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(rec) + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const int sb = c >> 1;     // ue8m0 scale byte of dims [32 sb, 32 sb + 32)
      const float s = ue ? ue8m0_to_f32(scw[sb >> 2] >> (8 * (sb & 3)))
                         : __uint_as_float(scw[c >> 3]);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        krow[16 * c + e] = e4m3_to_f32((w[e >> 2] >> (8 * (e & 3))) & 0xFFu) * s;
    }
  } else {
    const uint8_t *rec = record_ptr(L, sid);
    const uint4 s0 = __ldg(reinterpret_cast<const uint4 *>(rec + 256));
    const uint4 s1 = __ldg(reinterpret_cast<const uint4 *>(rec + 272));
    const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int c = j + 8 * kk;  // 16-byte chunk = dims [32c, 32c+32)
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(rec) + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int d = 32 * c + e;
        const int sb = d >> 4;  // scale byte index
        const float s = e4m3_to_f32((sw[sb >> 2] >> (8 * (sb & 3))) & 0xFFu);
        const uint32_t byte = (w[e >> 3] >> (8 * ((e >> 1) & 3))) & 0xFFu;
        const uint32_t nib = (e & 1) ? (byte >> 4) : (byte & 0xFu);
        krow[d] = e2m1_to_f32(nib) * s;
      }
    }
  }
  if (j == 0) {
    sm.valid[i] = ok ? 1 : 0;
    if (ok) {
      kept += 1;
      chk += row_hash(sid, r, lid);
    }
  }
}

template <int HPG>
__global__ void __launch_bounds__(kSimtThreads, 1) simt_decode_kernel(Params p) {
  pdl_launch_dependents();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem &sm = *reinterpret_cast<SimtSmem *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hg = blockIdx.x % p.HG;
  const int c = blockIdx.x / p.HG;
  int64_t u0, u1;   // live-balanced unit range (the Q area is free scratch here)
  cta_range(p, c, reinterpret_cast<int64_t *>(sm.q), u0, u1);
  if (u0 >= u1) return;
  const int32_t tf = (int32_t)(u0 / p.tpt), tl = (int32_t)((u1 - 1) / p.tpt);
  const int h0 = hg * HPG;
  constexpr int kPer = HPG * kD / kSimtThreads;  // accumulator elements per thread
  static_assert(kSimtThreads * 2 == kD, "accumulator layout assumes 2 dims per thread per head");

  for (int32_t t = tf; t <= tl; ++t) {
    const Segment seg = make_segment(p, c, t, u0, u1);
    // Q (fp32) with RoPE on dims 448..511 (NeoX or GPT-J pairs).
    int64_t pos = p.positions ? __ldg(p.positions + t) : 0;
    if (pos < 0 || (p.cos_sin && pos >= p.cs_rows)) {   // outside the table: flag, use row 0
      if (tid == 0) report_status(p.status, DSA_ERR_INVALID_ARG);
      pos = 0;
    }
    for (int e = tid; e < HPG * kD; e += kSimtThreads) {
      const int h = e / kD, d = e % kD;
      const __nv_bfloat16 *qh = p.q + (int64_t)t * p.q_st + (int64_t)(h0 + h) * p.q_sh;
      float x = __bfloat162float(qh[d]);
      if (p.cos_sin && d >= kRopeStart && p.rope_gptj) {   // pair (448+2i, 449+2i)
        const float *cs = p.cos_sin + pos * 64;
        const int i = (d - kRopeStart) >> 1;
        const float other = __bfloat162float(qh[d ^ 1]);
        x = (d & 1) ? x * cs[i] + other * cs[kRopeHalf + i] : x * cs[i] - other * cs[kRopeHalf + i];
      } else if (p.cos_sin && d >= kRopeStart) {
        const float *cs = p.cos_sin + pos * 64;
        if (d < kRopeStart + kRopeHalf) {
          const int i = d - kRopeStart;
          const float x2 = __bfloat162float(qh[d + kRopeHalf]);
          x = x * cs[i] - x2 * cs[kRopeHalf + i];
        } else {
          const int i = d - kRopeStart - kRopeHalf;
          const float x1 = __bfloat162float(qh[d - kRopeHalf]);
          x = x * cs[i] + x1 * cs[kRopeHalf + i];
        }
      }
      sm.q[e] = x;
    }
    if (tid < HPG) {
      sm.m[tid] = -INFINITY;
      sm.l[tid] = 0.f;
    }
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    uint32_t kept = 0, chk = 0;
    __syncthreads();

    for (int64_t u = seg.u_begin; u < seg.u_end; ++u) {
      int32_t lid, row0;
      unit_tile(p, u, lid, row0);
      const int32_t width = p.list[lid].width;
      for (int sub = 0; sub < kTile / kSub; ++sub) {
        const int32_t r0 = row0 + sub * kSub;
        if (r0 >= width) break;
        load_subtile(p, sm, lid, t, r0, kept, chk);
        __syncthreads();
        // Scores (log2 units): one warp per (head, row) pair, lanes over dims.
        for (int pi = warp; pi < HPG * kSub; pi += kSimtThreads / 32) {
          const int h = pi / kSub, r = pi % kSub;
          const float *qh = sm.q + h * kD;
          const float *kr = sm.k + r * kD;
          float a = 0.f;
#pragma unroll
          for (int kk = 0; kk < kD / 32; ++kk) a = fmaf(qh[lane + 32 * kk], kr[lane + 32 * kk], a);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
          if (lane == 0) sm.s[h * kSub + r] = sm.valid[r] ? a * p.scale_log2 : -INFINITY;
        }
        __syncthreads();
        // Online softmax per head.
        if (tid < HPG) {
          const int h = tid;
          float mt = -INFINITY;
          for (int r = 0; r < kSub; ++r) mt = fmaxf(mt, sm.s[h * kSub + r]);
          const float mo = sm.m[h];
          const float mn = fmaxf(mo, mt);
          float alpha = 1.f, sum = 0.f;
          if (mn != -INFINITY) {
            alpha = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
            for (int r = 0; r < kSub; ++r) {
              const float x = sm.s[h * kSub + r];
              const float pr = (x == -INFINITY) ? 0.f : exp2f(x - mn);
              sm.s[h * kSub + r] = pr;
              sum += pr;
            }
            sm.m[h] = mn;
            sm.l[h] = sm.l[h] * alpha + sum;
          } else {
            for (int r = 0; r < kSub; ++r) sm.s[h * kSub + r] = 0.f;
          }
          sm.alpha[h] = alpha;
        }
        __syncthreads();
        // O = O * alpha + P . K. Accumulator element i of this thread is
        // head i/2, dim tid + 256*(i%2).
#pragma unroll
        for (int i = 0; i < kPer; ++i) acc[i] *= sm.alpha[i >> 1];
#pragma unroll 1
        for (int r = 0; r < kSub; ++r) {
          const float k0 = sm.k[r * kD + tid], k1 = sm.k[r * kD + tid + 256];
#pragma unroll
          for (int i = 0; i < kPer; i += 2) {
            const float pr = sm.s[(i >> 1) * kSub + r];
            acc[i] = fmaf(pr, k0, acc[i]);
            acc[i + 1] = fmaf(pr, k1, acc[i + 1]);
          }
        }
        __syncthreads();
      }
    }

    // Row-selection record (head group 0 only).
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      kept += __shfl_xor_sync(0xffffffffu, kept, off);
      chk += __shfl_xor_sync(0xffffffffu, chk, off);
    }
    if (lane == 0) {
      sm.red[2 * warp] = (int32_t)kept;
      sm.red[2 * warp + 1] = (int32_t)chk;
    }
    __syncthreads();
    if (hg == 0 && tid == 0) {
      uint32_t k2 = 0, c2 = 0;
      for (int w = 0; w < kSimtThreads / 32; ++w) {
        k2 += (uint32_t)sm.red[2 * w];
        c2 += (uint32_t)sm.red[2 * w + 1];
      }
      int32_t *dst = seg.whole ? (p.sel + 2 * (int64_t)t) : (p.part_sel + 2 * (int64_t)seg.slot);
      dst[0] = (int32_t)k2;
      dst[1] = (int32_t)c2;
    }

    // Finalize: whole tokens -> out / lse with the sink; split -> partial slot.
    // MXFP8 output: whole tokens go to the fp32 staging area (cast later).
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int h = i >> 1, d = tid + 256 * (i & 1);
      const float l = sm.l[h], m = sm.m[h];
      if (seg.whole) {
        float v = 0.f;
        if (l > 0.f) {
          float den = l;
          if (p.sink) {
            const float sk = __ldg(p.sink + h0 + h);
            den = (sk == INFINITY) ? INFINITY : l + exp2f(sk * kLog2e - m);
          }
          v = acc[i] / den;
        }
        if (p.stage)
          p.stage[((int64_t)t * p.H + h0 + h) * kD + d] = v;
        else
          p.out[((int64_t)t * p.H + h0 + h) * kD + d] = __float2bfloat16_rn(v);
      } else {
        const int64_t slot = (int64_t)hg * 2 * p.C + seg.slot;
        p.part_o[(slot * HPG + h) * kD + d] = (l > 0.f) ? acc[i] / l : 0.f;
      }
    }
    if (tid < HPG) {
      const int h = tid;
      const float l = sm.l[h], m = sm.m[h];
      const float lse = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
      if (seg.whole)
        p.lse[(int64_t)t * p.H + h0 + h] = lse;
      else
        p.part_lse[((int64_t)hg * 2 * p.C + seg.slot) * HPG + h] = lse;
    }
    __syncthreads();
  }
}

}  // namespace dsa

namespace {
template <int N>
cudaError_t simt_setup(void *) {
  return cudaFuncSetAttribute(dsa::simt_decode_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(dsa::SimtSmem));
}
}  // namespace

cudaError_t dsa_launch_simt(const dsa::Params &p, cudaStream_t stream) {
  using namespace dsa;
  const size_t smem = sizeof(SimtSmem);
  const dim3 grid((unsigned)(p.C * p.HG)), block(kSimtThreads);
  cudaError_t err = cudaSuccess;
  switch (p.hpg) {
#define DSA_SIMT_CASE(N, BIT)                                                             \
  case N:                                                                                 \
    err = dsa_configure_once(BIT, &simt_setup<N>, nullptr);                               \
    if (err != cudaSuccess) return err;                                                   \
    simt_decode_kernel<N><<<grid, block, smem, stream>>>(p);                              \
    break;
    DSA_SIMT_CASE(16, 8)
    DSA_SIMT_CASE(32, 9)
    DSA_SIMT_CASE(48, 10)
    DSA_SIMT_CASE(64, 11)
#undef DSA_SIMT_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
