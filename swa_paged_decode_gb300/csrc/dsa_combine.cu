// dsa_combine.cu -- split-KV LSE combine.
//
// A token whose units the schedule spreads over CTAs c0..c1 left one
// normalised partial (O_i, lse_i) per CTA. This kernel merges them in CTA
// order (deterministic):
//   M = max_i lse_i, w_i = e^{lse_i - M} (0 for empty parts, lse_i = -inf),
//   out = sum_i w_i O_i / (sum_i w_i + e^{sink - M}),  lse = M + log sum_i w_i.
// Sources: the "production.py" page's Python KV merge (LSE-weighted
// normalised partials) and the vLLM swapab page's merge step (sink added to
// the denominator once; infinite sink or empty token gives zero output);
// FlashMLA's sparse_decode.h runs the same merge as a separate combine launch
// over o_accum / lse_accum.
//
// Grid: one block per (CTA boundary, head group). Boundary b (1 <= b < C)
// falls inside token t = b*upc / tpt; the block works only when b is the
// first boundary inside that token, so every split token is merged once.
#include "dsa_internal.cuh"

namespace dsa {

constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params p) {
  const int hg = blockIdx.x % p.HG;
  const int b = 1 + blockIdx.x / p.HG;
  const int64_t ub = (int64_t)b * p.upc;
  const int32_t t = (int32_t)(ub / p.tpt);
  const int64_t ts = (int64_t)t * p.tpt;
  if (ub == ts) return;                                  // boundary on a token start
  if (b > 1 && (int64_t)(b - 1) * p.upc > ts) return;    // not the first boundary in t
  const int32_t c0 = (int32_t)(ts / p.upc);
  const int32_t c1 = (int32_t)((ts + p.tpt - 1) / p.upc);
  const int hpg = p.hpg, h0 = hg * hpg;
  const int64_t slot_base = (int64_t)hg * 2 * p.C;

  // Row-selection record: sum of the parts (head group 0).
  if (hg == 0 && threadIdx.x == 0) {
    uint32_t k = 0, s = 0;
    for (int32_t c = c0; c <= c1; ++c) {
      const int32_t slot = 2 * c + (t == (int32_t)(cta_unit_begin(p, c) / p.tpt) ? 0 : 1);
      k += (uint32_t)p.part_sel[2 * slot];
      s += (uint32_t)p.part_sel[2 * slot + 1];
    }
    p.sel[2 * (int64_t)t] = (int32_t)k;
    p.sel[2 * (int64_t)t + 1] = (int32_t)s;
  }

  // Each thread: one head h and 4 consecutive dims per pass.
  for (int e = threadIdx.x; e < hpg * (kD / 4); e += kCombineThreads) {
    const int h = e / (kD / 4), d4 = e % (kD / 4);
    float mx = -INFINITY;
    for (int32_t c = c0; c <= c1; ++c) {
      const int32_t slot = 2 * c + (t == (int32_t)(cta_unit_begin(p, c) / p.tpt) ? 0 : 1);
      mx = fmaxf(mx, p.part_lse[(slot_base + slot) * hpg + h]);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float z = 0.f;
    if (mx != -INFINITY) {
      for (int32_t c = c0; c <= c1; ++c) {
        const int32_t slot = 2 * c + (t == (int32_t)(cta_unit_begin(p, c) / p.tpt) ? 0 : 1);
        const float li = p.part_lse[(slot_base + slot) * hpg + h];
        if (li == -INFINITY) continue;
        const float w = expf(li - mx);
        const float4 o = reinterpret_cast<const float4 *>(
            p.part_o + ((slot_base + slot) * hpg + h) * kD)[d4];
        z += w;
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
      }
    }
    float inv = 0.f;
    if (z > 0.f) {
      float den = z;
      if (p.sink) {
        const float sk = __ldg(p.sink + h0 + h);
        den = (sk == INFINITY) ? INFINITY : z + expf(sk - mx);
      }
      inv = 1.f / den;
    }
    __nv_bfloat16 *o = p.out + ((int64_t)t * p.H + h0 + h) * kD + 4 * d4;
    __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 c2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&a);
    pk.y = *reinterpret_cast<uint32_t *>(&c2);
    *reinterpret_cast<uint2 *>(o) = pk;
    if (d4 == 0) p.lse[(int64_t)t * p.H + h0 + h] = (z > 0.f) ? mx + logf(z) : -INFINITY;
  }
}

}  // namespace dsa

cudaError_t dsa_launch_combine(const dsa::Params &p, cudaStream_t stream) {
  using namespace dsa;
  if (p.C <= 1) return cudaSuccess;
  const dim3 grid((unsigned)((p.C - 1) * p.HG)), block(kCombineThreads);
  combine_kernel<<<grid, block, 0, stream>>>(p);
  return cudaGetLastError();
}
