// dsa_combine.cu -- split-KV LSE combine, and the MXFP8 output cast of the
// V4.1 form (mx_epilogue_kernel, below).
//
// A token whose units the schedule spreads over CTAs c0..c1 left one
// normalised partial (O_i, lse_i) per CTA. This kernel merges them in a
// fixed order (deterministic, independent of timing):
//   M = max_i lse_i, w_i = e^{lse_i - M} (0 for empty parts, lse_i = -inf),
//   out = sum_i w_i O_i / (sum_i w_i + e^{sink - M}),  lse = M + log sum_i w_i.
// Sources: the "production.py" page's Python KV merge (LSE-weighted
// normalised partials) and the vLLM swapab page's merge step (sink added to
// the denominator once; infinite sink or empty token gives zero output);
// FlashMLA's sparse_decode.h runs the same merge as a separate combine launch
// over o_accum / lse_accum.
//
// Grid: x = one block per (CTA boundary, head group), y = chunks of 8 heads
// x S slices of the dims (S = 16 when a token can span 8 or more CTAs,
// else 4).
// Boundary b (1 <= b < C) is the first unit bounds[b] of CTA b (ranges set
// by the run kernel); it falls inside token t = bounds[b] / tpt and its
// blocks work only when b is the first boundary inside that token, so every
// split token is merged once, by hpg/8 * S blocks per head group. A block
// first turns the parts' lse into weights in shared memory (one warp per
// head), then streams the partial O.
#include "dsa_internal.cuh"

namespace dsa {

constexpr int kCombineThreads = 256;
constexpr int kCombineHeads = 8;    // heads per block: one warp per head for the weights
constexpr int kCombineLoads = 8;    // partial O loads of a thread in flight together

// S dim slices per chunk of 8 heads (grid y = hpg/8 * S). A block covers 8
// heads x 512/S dims: I = 8 * 128/S float4 items. With I >= 256 a thread
// sums K = I/256 items over all parts; with I < 256 its 256 threads form
// G = 256/I groups, group g summing parts g, g + G, ... of every item, so a
// token split into many parts keeps G times more loads in flight per item.
// Groups are added in group order: the result does not depend on timing.
template <int S>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params p) {
  constexpr int kQ4 = kD / 4 / S;                         // float4s per head in a slice
  constexpr int kI = kCombineHeads * kQ4;
  constexpr int kG = kI >= kCombineThreads ? 1 : kCombineThreads / kI;
  constexpr int kK = kI >= kCombineThreads ? kI / kCombineThreads : 1;
  constexpr int kU = kCombineLoads / kK;                 // parts per round
  extern __shared__ float cs[];   // w[nparts][8], inv[8], then (G-1) x I float4
  pdl_wait_primary();   // the decode kernel's partials are complete and visible
  const int hg = blockIdx.x % p.HG;
  const int b = 1 + blockIdx.x / p.HG;
  // even split: CTA b starts at unit b * upc (no load needed to leave early)
  const int64_t ub = p.balance ? __ldg(p.bounds + b)
                               : ((int64_t)b * p.upc < p.U ? (int64_t)b * p.upc : p.U);
  if (ub >= p.U) return;                                 // empty CTAs at the end
  const int32_t t = (int32_t)(ub / p.tpt);
  const int64_t ts = (int64_t)t * p.tpt, te = ts + p.tpt;
  if (ub == ts) return;                                  // boundary on a token start
  if (b > 1) {                                           // not the first boundary in t
    const int64_t up = p.balance ? __ldg(p.bounds + b - 1) : (int64_t)(b - 1) * p.upc;
    if (up > ts) return;
  }
  // parts: CTA b-1 (holds unit ts) through the CTA holding unit te-1
  const int32_t c0 = b - 1;
  int32_t c1;
  bool c0_late;
  if (!p.balance) {   // even split: the CTA holding unit te-1 directly
    const int64_t cl = (te - 1) / p.upc;
    c1 = (int32_t)(cl < p.C - 1 ? cl : p.C - 1);
    c0_late = (int64_t)c0 * p.upc < ts;
  } else {            // balanced ranges: a token spans a few CTAs at most
    c1 = b;
    while (c1 + 1 < p.C && __ldg(p.bounds + c1 + 1) < te) ++c1;
    c0_late = __ldg(p.bounds + c0) < ts;
  }
  const int np = c1 - c0 + 1;
  const int hpg = p.hpg, h0 = hg * hpg, hb = ((int)blockIdx.y / S) * kCombineHeads;
  const int slice = (int)blockIdx.y % S;
  const int64_t slot_base = (int64_t)hg * 2 * p.C;
  // Partial slot of CTA c for token t: 2c when t is the CTA's first token,
  // else 2c + 1 (only the first CTA of the token can start in an earlier one).
  auto slot_of = [&](int32_t c) -> int64_t { return 2 * (int64_t)c + ((c == c0 && c0_late) ? 1 : 0); };
  float *w_s = cs;
  float *inv_s = cs + np * kCombineHeads;
  float4 *red_s = reinterpret_cast<float4 *>(cs + (np + 1) * kCombineHeads);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t part_n = (int64_t)p.HG * 2 * p.C * hpg;   // partial (slot, head) records

  // Weights, one warp per head: M = max_i lse_i, w_i = e^{lse_i - M},
  // z = sum_i w_i (lanes over the parts, then a butterfly).
  {
    const int h = warp;
    float mx = -INFINITY;
    for (int q = lane; q < np; q += 32) {
      const int64_t ip = (slot_base + slot_of(c0 + q)) * hpg + hb + h;
      const float li = dbg_ok(p.status, ip >= 0 && ip < part_n, kDbgPartial) ? p.part_lse[ip] : -INFINITY;
      w_s[q * kCombineHeads + h] = li;
      mx = fmaxf(mx, li);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float z = 0.f;
    for (int q = lane; q < np; q += 32) {
      const float li = w_s[q * kCombineHeads + h];
      const float w = (li == -INFINITY) ? 0.f : expf(li - mx);
      w_s[q * kCombineHeads + h] = w;
      z += w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (lane == 0) {
      float inv = 0.f;
      if (z > 0.f) {
        float den = z;
        if (p.sink) {
          const float sk = __ldg(p.sink + h0 + hb + h);
          den = (sk == INFINITY) ? INFINITY : z + expf(sk - mx);
        }
        inv = 1.f / den;
      }
      inv_s[h] = inv;
      const int64_t il = (int64_t)t * p.H + h0 + hb + h;
      if (slice == 0 && dbg_ok(p.status, il >= 0 && il < (int64_t)p.T * p.H, kDbgOut))
        p.lse[il] = (z > 0.f) ? mx + logf(z) : -INFINITY;
    }
  }
  // Row-selection record: sum of the parts (one block per token, warp 0).
  if (hg == 0 && blockIdx.y == 0 && warp == 0 &&
      dbg_ok(p.status, t >= 0 && t < p.T && c0 >= 0 && c1 < p.C, kDbgSel)) {
    uint32_t k = 0, s2 = 0;
    for (int q = lane; q < np; q += 32) {
      const int64_t slot = slot_of(c0 + q);
      k += (uint32_t)p.part_sel[2 * slot];
      s2 += (uint32_t)p.part_sel[2 * slot + 1];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      k += __shfl_xor_sync(0xffffffffu, k, off);
      s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    }
    if (lane == 0) {
      p.sel[2 * (int64_t)t] = (int32_t)k;
      p.sel[2 * (int64_t)t + 1] = (int32_t)s2;
    }
  }
  __syncthreads();

  // out = sum_i w_i O_i * inv. Item e: one head, 4 consecutive dims of the
  // slice. A thread takes items e_k = (tid % I) + 256 k and parts g, g + G, ...
  const int g = tid / (kI < kCombineThreads ? kI : kCombineThreads);
  float4 acc[kK];
#pragma unroll
  for (int k = 0; k < kK; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = g; q0 < np; q0 += kG * kU) {
    float4 o[kU][kK];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = q0 + u * kG;
#pragma unroll
      for (int k = 0; k < kK; ++k) {
        const int e = (tid % (kI < kCombineThreads ? kI : kCombineThreads)) + kCombineThreads * k;
        const int h = e / kQ4, d4 = slice * kQ4 + e % kQ4;
        o[u][k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q < np && w_s[q * kCombineHeads + h] != 0.f) {
          const int64_t ip = (slot_base + slot_of(c0 + q)) * hpg + hb + h;
          if (dbg_ok(p.status, ip >= 0 && ip < part_n, kDbgPartial))
            o[u][k] = __ldg(reinterpret_cast<const float4 *>(p.part_o + ip * kD) + d4);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = q0 + u * kG;
#pragma unroll
      for (int k = 0; k < kK; ++k) {
        const int e = (tid % (kI < kCombineThreads ? kI : kCombineThreads)) + kCombineThreads * k;
        const int h = e / kQ4;
        const float w = q < np ? w_s[q * kCombineHeads + h] : 0.f;
        if (w == 0.f) continue;
        acc[k].x = fmaf(w, o[u][k].x, acc[k].x);
        acc[k].y = fmaf(w, o[u][k].y, acc[k].y);
        acc[k].z = fmaf(w, o[u][k].z, acc[k].z);
        acc[k].w = fmaf(w, o[u][k].w, acc[k].w);
      }
    }
  }
  if constexpr (kG > 1) {   // groups 1.. hand their sums to group 0, added in group order
    const int e = tid % kI;
    if (g > 0) red_s[(g - 1) * kI + e] = acc[0];
    __syncthreads();
    if (g > 0) return;
#pragma unroll
    for (int k = 0; k < kG - 1; ++k) {
      const float4 r = red_s[k * kI + e];
      acc[0].x += r.x;
      acc[0].y += r.y;
      acc[0].z += r.z;
      acc[0].w += r.w;
    }
  }
#pragma unroll
  for (int k = 0; k < kK; ++k) {
    const int e = (tid % (kI < kCombineThreads ? kI : kCombineThreads)) + kCombineThreads * k;
    const int h = e / kQ4, d4 = slice * kQ4 + e % kQ4;
    const float inv = inv_s[h];
    const int64_t io = ((int64_t)t * p.H + h0 + hb + h) * kD + 4 * d4;
    if (!dbg_ok(p.status, io >= 0 && io + 4 <= (int64_t)p.T * p.H * kD, kDbgOut)) continue;
    if (p.stage) {   // MXFP8 output: fp32 to the staging area, cast later
      *reinterpret_cast<float4 *>(p.stage + io) =
          make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
      continue;
    }
    __nv_bfloat162 a = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
    __nv_bfloat162 c2 = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&a);
    pk.y = *reinterpret_cast<uint32_t *>(&c2);
    *reinterpret_cast<uint2 *>(p.out + io) = pk;
  }
}

// ------------------------------------------------------------ MXFP8 cast
// The V4.1 output epilogue (the swapab page's merge step): per token, head
// and 32-dim chunk, the inverse GPT-J rotation of dims >= 448 (table row of
// the token's position; pairs lie inside a thread's 4 dims), an ue8m0 scale
// E = ceil(log2(max(amax, 1e-10) * fp32(1/448))) + 127 and e4m3 codes of
// x * 2^(127 - E) (round to nearest even, saturating), o-fused layout.
// A warp takes kMxUnits consecutive (token, head, 128-dim quarter) units;
// 8 lanes = one 32-dim chunk.
constexpr int kMxThreads = 256;
constexpr int kMxUnits = 4;   // units per warp, their loads in flight together

__global__ void __launch_bounds__(kMxThreads) mx_epilogue_kernel(Params p) {
  pdl_wait_primary();   // the staged outputs are complete and visible
  const int64_t units = (int64_t)p.T * p.H * 4;
  const int64_t w0 = ((int64_t)blockIdx.x * (kMxThreads / 32) + (threadIdx.x >> 5)) * kMxUnits;
  const int lane = threadIdx.x & 31;
  // the warp's units' 512-byte rows, loaded together (kMxUnits in flight)
  float4 v[kMxUnits];
#pragma unroll
  for (int i = 0; i < kMxUnits; ++i) {
    const int64_t unit = w0 + i;
    v[i] = unit < units
               ? __ldg(reinterpret_cast<const float4 *>(p.stage + (unit >> 2) * kD + 128 * (unit & 3)) + lane)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int i = 0; i < kMxUnits; ++i) {
    const int64_t unit = w0 + i;
    if (unit >= units) break;   // whole warps leave together
    const int quarter = (int)(unit & 3);
    const int64_t th = unit >> 2;
    const int64_t t = th / p.H;
    const int h = (int)(th - t * p.H);
    const int d0 = 128 * quarter + 4 * lane;
    float x[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    const float *cs_row = mx_rope_row(p, t);
    if (cs_row != nullptr && d0 >= kRopeStart) {
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        const int k = (d0 - kRopeStart) / 2 + pr;
        const float c = __ldg(cs_row + k), sn = __ldg(cs_row + kRopeHalf + k);
        const float oe = x[2 * pr], oo = x[2 * pr + 1];
        x[2 * pr] = fmaf(oe, c, sn * oo);
        x[2 * pr + 1] = fmaf(oo, c, -(sn * oe));
      }
    }
    float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    const uint32_t E = ue8m0_ceil(fmaxf(a, 1e-10f) * (1.0f / 448.0f));
    const float sc = ue8m0_inverse(E);
    const uint32_t codes =
        e4m3x2_rn_sat(x[0] * sc, x[1] * sc) | (e4m3x2_rn_sat(x[2] * sc, x[3] * sc) << 16);
    const int c = d0 >> 5;
    *reinterpret_cast<uint32_t *>(mx_chunk(p, t, h, c) + (d0 & 31)) = codes;
    if ((d0 & 31) == 0) *mx_scale_byte(p, t, h, c) = (uint8_t)E;
  }
}

}  // namespace dsa

namespace {
template <int S>
cudaError_t combine_setup(void *) {
  return cudaFuncSetAttribute(dsa::combine_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              227 * 1024);
}

template <int S>
cudaError_t launch_combine(const dsa::Params &p, cudaStream_t stream, int64_t np_max, int bit) {
  using namespace dsa;
  constexpr int kI = kCombineHeads * (kD / 4 / S);
  constexpr int kG = kI >= kCombineThreads ? 1 : kCombineThreads / kI;
  const size_t smem = (size_t)(np_max + 1) * kCombineHeads * sizeof(float) +
                      (size_t)(kG - 1) * kI * sizeof(float4);
  if (smem > 48 * 1024) {   // raised once per device to the largest opt-in size
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    const cudaError_t e = dsa_configure_once(bit, &combine_setup<S>, nullptr);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)((p.C - 1) * p.HG), (unsigned)(p.hpg / kCombineHeads * S)),
      block(kCombineThreads);
  // Launched as a programmatic dependent of the decode kernel before it on
  // the stream: its blocks may be scheduled while that kernel drains.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<S>, p);
}
}  // namespace

cudaError_t dsa_launch_combine(const dsa::Params &p, cudaStream_t stream) {
  if (p.C <= 1) return cudaSuccess;
  // A token spans at most min(C, tpt + 1) CTAs; on average about
  // tpt / upc + 1. Few parts: blocks of 8 whole heads (fewer, larger
  // blocks); many parts: 16 slices, 4 thread groups over the parts.
  const int64_t np_max = p.C < (int64_t)p.tpt + 1 ? p.C : (int64_t)p.tpt + 1;
  const int64_t np_avg = (p.tpt + p.upc - 1) / (p.upc > 0 ? p.upc : 1) + 1;
  if (np_avg <= 4) return launch_combine<1>(p, stream, np_max, 16);
  if (np_avg < 16) return launch_combine<4>(p, stream, np_max, 17);
  return launch_combine<16>(p, stream, np_max, 18);
}

cudaError_t dsa_launch_mx_epilogue(const dsa::Params &p, cudaStream_t stream) {
  using namespace dsa;
  const int64_t units = (int64_t)p.T * p.H * 4;
  if (units == 0) return cudaSuccess;
  const int64_t per_block = (int64_t)(kMxThreads / 32) * kMxUnits;
  const int64_t blocks = (units + per_block - 1) / per_block;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  // Programmatic dependent of the kernel before it (combine, or the decode
  // kernel when nothing was split): it waits for that grid's completion.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kMxThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mx_epilogue_kernel, p);
}
