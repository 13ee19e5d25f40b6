// dsa_api.cu -- the C ABI (include/dsa_decode.h): planning, argument
// validation and launches. Host code only; kernels live in the other
// translation units.
//
// Validation mirrors the checks FlashMLA's sparse_attn_decode_interface
// (csrc/api/sparse_decode.h page) makes before launching: MQA with head dim
// 512, extra indices present iff an extra cache is present, record-sized
// contiguous pages, dtype/shape of every optional input.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "dsa_internal.cuh"

using dsa::Params;

namespace {
constexpr int kCfgDevices = 64;
std::mutex g_cfg_mutex;
uint64_t g_cfg_done[kCfgDevices] = {};   // per device: bit i = variant i set up
}  // namespace

cudaError_t dsa::dsa_configure_once(int bit, cudaError_t (*f)(void *), void *arg) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kCfgDevices || bit < 0 || bit >= 64) return f(arg);
  std::lock_guard<std::mutex> lock(g_cfg_mutex);
  if (g_cfg_done[dev] & (1ull << bit)) return cudaSuccess;
  e = f(arg);
  if (e == cudaSuccess) g_cfg_done[dev] |= 1ull << bit;
  return e;
}

namespace {

// NVTX range over one entry point (host side: argument checks and launches),
// so a profiler timeline shows each run / combine call.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

constexpr int64_t kAlignWs = 256;
constexpr int64_t kStatusBytes = 256;

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
int record_bytes(int32_t fmt) {
  if (fmt == DSA_REC_FP8_528 || fmt == DSA_REC_FP8_528_UE8M0) return 528;
  if (fmt == DSA_REC_MODEL1_584) return 584;
  if (fmt == DSA_REC_V32_656) return 656;
  return fmt == DSA_REC_NVFP4_288 ? 288 : -1;
}

bool heads_supported(int32_t H) {
  return H == 16 || H == 32 || H == 48 || H == 64 || H == 96 || H == 128;
}

dsa_status fill_list(const dsa_cache_desc *c, const int32_t *idx, int64_t stride,
                     const int32_t *lens, int32_t width, dsa::ListArgs &L) {
  if (!c || !idx || !lens || !c->base) return DSA_ERR_INVALID_ARG;
  const int rb = record_bytes(c->format);
  if (rb < 0) return DSA_ERR_UNSUPPORTED;
  if (c->num_pages < 1 || !pow2(c->page_size)) return DSA_ERR_INVALID_ARG;
  if (c->page_stride_bytes < (int64_t)c->page_size * rb) return DSA_ERR_INVALID_ARG;
  if (c->num_pages * (int64_t)c->page_size > (int64_t)INT32_MAX + 1) return DSA_ERR_UNSUPPORTED;
  if (stride < width) return DSA_ERR_INVALID_ARG;
  if (!aligned(c->base, 16) || c->page_stride_bytes % 16 != 0) return DSA_ERR_ALIGNMENT;
  if (!aligned(idx, 4) || !aligned(lens, 4)) return DSA_ERR_ALIGNMENT;
  L.base = static_cast<const uint8_t *>(c->base);
  L.num_slots = c->num_pages * (int64_t)c->page_size;
  L.page_stride = c->page_stride_bytes;
  L.ids = idx;
  L.lens = lens;
  L.idx_stride = stride;
  int sh = 0;
  while ((1 << sh) < c->page_size) ++sh;
  L.page_shift = sh;
  L.page_mask = c->page_size - 1;
  L.fmt = c->format;
  L.rec = rb;
  L.width = width;
  L.tiles = (width + dsa::kTile - 1) / dsa::kTile;
  L.extent = c->num_pages * c->page_stride_bytes;
#ifdef DSA_DEBUG
  // Checking build only: a smaller extent for the record checks (a test
  // knob: records past it are reported and skipped, never read).
  if (const char *cap = std::getenv("DSA_DEBUG_CHECK_EXTENT")) {
    const long long v = std::atoll(cap);
    if (v > 0 && v < L.extent) L.extent = v;
  }
#endif
  L.aligned32 = (aligned(c->base, 32) && c->page_stride_bytes % 32 == 0 && rb % 32 == 0) ? 1 : 0;
  L.sectors32 = (aligned(c->base, 32) && c->page_stride_bytes % 32 == 0) ? 1 : 0;
  return DSA_OK;
}

bool plan_ok(const dsa_decode_plan_t *plan) {
  return plan && plan->magic == dsa::kPlanMagic && plan->abi_version == DSA_DECODE_ABI_VERSION;
}

void fill_schedule(const dsa_decode_plan_t *plan, void *ws, Params &p) {
  p.T = plan->num_tokens;
  p.H = plan->num_heads;
  p.hpg = plan->heads_per_group;
  p.HG = plan->head_groups;
  p.tpt = plan->tiles_per_token;
  p.upc = plan->units_per_cta;
  p.C = plan->ctas_per_group;
  p.U = plan->total_units;
  char *w = static_cast<char *>(ws);
  p.status = reinterpret_cast<int32_t *>(w);
  p.sel = reinterpret_cast<int32_t *>(w + plan->ws_sel_offset);
  p.part_lse = reinterpret_cast<float *>(w + plan->ws_part_lse_offset);
  p.part_sel = reinterpret_cast<int32_t *>(w + plan->ws_part_sel_offset);
  p.part_o = reinterpret_cast<float *>(w + plan->ws_part_o_offset);
  p.bounds = reinterpret_cast<int64_t *>(w + plan->ws_bounds_offset);
  p.balance = (int32_t)plan->balance_live;
  p.wait_budget = plan->wait_budget_cycles > 0 ? (long long)plan->wait_budget_cycles : 0;
  p.pq = plan->producer_q != 0 ? 1 : 0;
  p.merge = plan->merge_in_run != 0 ? 1 : 0;
  p.tok_cnt = reinterpret_cast<int32_t *>(w + plan->ws_count_offset);
}

dsa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// Output options shared by run and combine: bf16 `out` or the MXFP8
// descriptor, the RoPE pairing and the inverse-rotation rule.
dsa_status fill_output(const dsa_decode_plan_t *plan, const int64_t *positions,
                       const float *cos_sin, int64_t cos_sin_rows, int32_t rope_style, void *out,
                       const dsa_mxfp8_out *mx, Params &p) {
  if (rope_style != DSA_ROPE_NEOX && rope_style != DSA_ROPE_GPTJ) return DSA_ERR_INVALID_ARG;
  if ((out == nullptr) == (mx == nullptr)) return DSA_ERR_INVALID_ARG;
  p.rope_gptj = rope_style == DSA_ROPE_GPTJ ? 1 : 0;
  p.positions = positions;
  p.cos_sin = cos_sin;
  p.cs_rows = cos_sin_rows;
  if (out) {
    if (!aligned(out, 16)) return DSA_ERR_ALIGNMENT;
    p.out = static_cast<__nv_bfloat16 *>(out);
    return DSA_OK;
  }
  if (!mx->data || !mx->scale || mx->group_size < 1 || plan->num_heads % mx->group_size != 0)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(mx->data, 4) || mx->data_stride_t % 4 != 0 || mx->data_stride_g % 4 != 0 ||
      !aligned(mx->scale, 4))
    return DSA_ERR_ALIGNMENT;
  if (cos_sin && rope_style == DSA_ROPE_NEOX) return DSA_ERR_UNSUPPORTED;
  p.mx_on = 1;
  p.mx_g = mx->group_size;
  p.mx_data = static_cast<uint8_t *>(mx->data);
  p.mx_scale = reinterpret_cast<uint8_t *>(mx->scale);
  p.mx_st = mx->data_stride_t;
  p.mx_sg = mx->data_stride_g;
  p.mx_sst = mx->scale_stride_t;
  p.mx_ssg = mx->scale_stride_g;
  p.mx_ssw = mx->scale_stride_w;
  return DSA_OK;
}

dsa_status run_impl(const dsa_decode_plan_t *plan, void *workspace, size_t workspace_bytes,
                    const void *q, int64_t q_stride_t, int64_t q_stride_h,
                    const dsa_cache_desc *swa_cache, const int32_t *swa_idx,
                    int64_t swa_idx_stride, const int32_t *swa_lens,
                    const dsa_cache_desc *extra_cache, const int32_t *extra_idx,
                    int64_t extra_idx_stride, const int32_t *extra_lens, const float *sink,
                    const int64_t *positions, const float *cos_sin, int64_t cos_sin_rows,
                    int32_t rope_style, float scale, void *out, const dsa_mxfp8_out *mx,
                    float *lse, dsa_stream_t stream) {
  if (!plan_ok(plan)) return DSA_ERR_PLAN;
  if (plan->num_tokens == 0) return DSA_OK;
  if (!q || !lse) return DSA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return DSA_ERR_INVALID_ARG;
  const int64_t dqk = plan->d_qk == 576 ? 576 : dsa::kD;
  if (q_stride_h < dqk || q_stride_t < (int64_t)plan->num_heads * q_stride_h)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || q_stride_t % 8 != 0 || q_stride_h % 8 != 0) return DSA_ERR_ALIGNMENT;
  if (!aligned(lse, 4)) return DSA_ERR_ALIGNMENT;
  const bool has_extra = plan->extra_width > 0;
  if (has_extra != (extra_cache != nullptr) || has_extra != (extra_idx != nullptr) ||
      has_extra != (extra_lens != nullptr))
    return DSA_ERR_INVALID_ARG;
  if ((positions == nullptr) != (cos_sin == nullptr)) return DSA_ERR_INVALID_ARG;
  if (cos_sin && (cos_sin_rows < 1 || !aligned(cos_sin, 16) || !aligned(positions, 8)))
    return cos_sin_rows < 1 ? DSA_ERR_INVALID_ARG : DSA_ERR_ALIGNMENT;
  if (sink && !aligned(sink, 4)) return DSA_ERR_ALIGNMENT;
  const int64_t need = mx ? plan->workspace_bytes_mx : plan->workspace_bytes;
  if (!workspace || (int64_t)workspace_bytes < need || !aligned(workspace, kAlignWs))
    return DSA_ERR_WORKSPACE;

  Params p;
  std::memset(&p, 0, sizeof(p));
  dsa_status s = fill_output(plan, positions, cos_sin, cos_sin_rows, rope_style, out, mx, p);
  if (s != DSA_OK) return s;
  if (p.mx_on) p.stage = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan->ws_stage_offset);
  s = fill_list(swa_cache, swa_idx, swa_idx_stride, swa_lens, plan->swa_width, p.list[0]);
  if (s != DSA_OK) return s;
  p.nlists = 1;
  if (has_extra) {
    s = fill_list(extra_cache, extra_idx, extra_idx_stride, extra_lens, plan->extra_width,
                  p.list[1]);
    if (s != DSA_OK) return s;
    p.nlists = 2;
  }
  // V3.2 records: in every list, with a plan for 576-dim keys, no RoPE
  // table and no V4.1 output options; other records with 512-dim keys
  for (int i = 0; i < p.nlists; ++i)
    if ((p.list[i].fmt == DSA_REC_V32_656) != (dqk == 576)) return DSA_ERR_UNSUPPORTED;
  if (dqk == 576 && (cos_sin || mx || rope_style != DSA_ROPE_NEOX)) return DSA_ERR_UNSUPPORTED;
  p.dqk = (int32_t)dqk;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.q_st = q_stride_t;
  p.q_sh = q_stride_h;
  p.sink = sink;
  p.scale = scale;
  p.scale_log2 = scale * dsa::kLog2e;
  p.lse = lse;
  fill_schedule(plan, workspace, p);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // status word and the per-token unit counts of the in-run merge: one memset
  cudaError_t e = cudaMemsetAsync(workspace, 0, (size_t)plan->ws_sel_offset, st);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  return cuda_status(plan->kernel == dsa::kKernelTc ? dsa_launch_tc(p, st)
                                                    : dsa_launch_simt(p, st));
}

dsa_status combine_impl(const dsa_decode_plan_t *plan, void *workspace, size_t workspace_bytes,
                        const float *sink, const int64_t *positions, const float *cos_sin,
                        int64_t cos_sin_rows, int32_t rope_style, void *out,
                        const dsa_mxfp8_out *mx, float *lse, dsa_stream_t stream) {
  if (!plan_ok(plan)) return DSA_ERR_PLAN;
  // bf16 output: only split tokens need this call; MXFP8: every token does
  if (plan->num_tokens == 0 || (!mx && plan->split_tokens == 0)) return DSA_OK;
  if (!lse) return DSA_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || (sink && !aligned(sink, 4))) return DSA_ERR_ALIGNMENT;
  if ((positions == nullptr) != (cos_sin == nullptr)) return DSA_ERR_INVALID_ARG;
  if (cos_sin && (cos_sin_rows < 1 || !aligned(cos_sin, 16) || !aligned(positions, 8)))
    return cos_sin_rows < 1 ? DSA_ERR_INVALID_ARG : DSA_ERR_ALIGNMENT;
  const int64_t need = mx ? plan->workspace_bytes_mx : plan->workspace_bytes;
  if (!workspace || (int64_t)workspace_bytes < need || !aligned(workspace, kAlignWs))
    return DSA_ERR_WORKSPACE;
  Params p;
  std::memset(&p, 0, sizeof(p));
  dsa_status s = fill_output(plan, positions, cos_sin, cos_sin_rows, rope_style, out, mx, p);
  if (s != DSA_OK) return s;
  fill_schedule(plan, workspace, p);
  p.list[0].tiles = plan->tiles_swa;
  p.list[1].tiles = plan->tiles_extra;
  p.sink = sink;
  p.lse = lse;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (p.mx_on) p.stage = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan->ws_stage_offset);
  // (a plan whose run kernel merged the split tokens launches no merge here)
  cudaError_t e = plan->merge_in_run ? cudaSuccess : dsa_launch_combine(p, st);
  if (e == cudaSuccess && p.mx_on) e = dsa_launch_mx_epilogue(p, st);
  return cuda_status(e);
}

}  // namespace

extern "C" {

int32_t dsa_decode_abi_version(void) { return DSA_DECODE_ABI_VERSION; }

const char *dsa_decode_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case DSA_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case DSA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case DSA_ERR_CUDA: return "CUDA runtime error";
    case DSA_ERR_TIMEOUT: return "device wait timed out";
    case DSA_ERR_PLAN: return "invalid or mismatched plan";
    case DSA_ERR_BOUNDS: return "checking build: an out-of-extent access was skipped";
  }
  return "unknown status";
}

dsa_status dsa_decode_plan(int32_t num_tokens, int32_t num_heads, int32_t swa_width,
                           int32_t extra_width, int32_t num_sms, dsa_decode_plan_t *plan,
                           size_t *workspace_bytes) {
  return dsa_decode_plan_qk(num_tokens, num_heads, swa_width, extra_width, num_sms, 512, plan,
                            workspace_bytes);
}

dsa_status dsa_decode_plan_qk(int32_t num_tokens, int32_t num_heads, int32_t swa_width,
                              int32_t extra_width, int32_t num_sms, int32_t d_qk,
                              dsa_decode_plan_t *plan, size_t *workspace_bytes) {
  if (!plan || !workspace_bytes) return DSA_ERR_INVALID_ARG;
  if (num_tokens < 0 || swa_width < 1 || extra_width < 0 || num_sms < 0)
    return DSA_ERR_INVALID_ARG;
  if (d_qk != 512 && d_qk != 576) return DSA_ERR_INVALID_ARG;
  if (!heads_supported(num_heads)) return DSA_ERR_UNSUPPORTED;
  // 576-dim keys: groups of at most 32 heads on the tensor-core kernel
  if (d_qk == 576 && (num_heads == 48 || num_heads == 96)) return DSA_ERR_UNSUPPORTED;
  if (num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DSA_ERR_CUDA;
  }
  std::memset(plan, 0, sizeof(*plan));
  plan->magic = dsa::kPlanMagic;
  plan->abi_version = DSA_DECODE_ABI_VERSION;
  plan->num_tokens = num_tokens;
  plan->num_heads = num_heads;
  plan->swa_width = swa_width;
  plan->extra_width = extra_width;
  plan->num_sms = num_sms;
  plan->d_qk = d_qk;
  plan->head_groups = num_heads <= 64 ? 1 : 2;
  plan->heads_per_group = num_heads / plan->head_groups;
  while (d_qk == 576 && plan->heads_per_group > 32) {
    plan->head_groups *= 2;
    plan->heads_per_group /= 2;
  }
  plan->tiles_swa = (swa_width + dsa::kTile - 1) / dsa::kTile;
  plan->tiles_extra = (extra_width + dsa::kTile - 1) / dsa::kTile;
  plan->tiles_per_token = plan->tiles_swa + plan->tiles_extra;
  plan->total_units = (int64_t)num_tokens * plan->tiles_per_token;
  // Tensor-core kernel for 16/32/64 heads per group; the CUDA-core kernel
  // takes 48/96 heads, or any shape when DSA_DECODE_KERNEL=simt is set (a
  // cross-check switch read only here, at planning time).
  plan->kernel = dsa_tc_supports(plan->heads_per_group) ? dsa::kKernelTc : dsa::kKernelSimt;
  if (const char *k = std::getenv("DSA_DECODE_KERNEL"))
    if (std::strcmp(k, "simt") == 0) plan->kernel = dsa::kKernelSimt;
  // Small batches: halve the heads per group (down to 16) while the units of
  // all head groups would give each SM at most 4 (the first halving) or 2
  // (further ones). Each CTA then stages Q for and finalizes fewer heads --
  // the per-token steps that bound a CTA with a few tiles -- and more CTAs
  // share them; the groups read the same records (the repeats mostly hit
  // L2). Measured per step: config 5 T=1 53 -> 29 us, T=8 60 -> 45 us,
  // config 2 39 -> 31 us, larger batches unchanged. FlashMLA spreads a small
  // batch the same way over num_sm_parts = num_sms / s_q parts
  // (sparse_decode.h, get_meta); here the extra parts split the heads.
  if (plan->kernel == dsa::kKernelTc) {
    const int32_t hpg0 = plan->heads_per_group;
    while (plan->heads_per_group > 16 &&
           plan->total_units * plan->head_groups <=
               (plan->heads_per_group == hpg0 ? 4 : 2) * (int64_t)num_sms) {
      plan->head_groups *= 2;
      plan->heads_per_group /= 2;
    }
  }
  // Grid: as many CTAs per head group as an even split of the units needs
  // (FlashMLA's num_sm_parts idea, sparse_decode.h get_meta). The run kernel
  // then places the CTA boundaries so that each CTA gets the same number of
  // live tiles (lengths are read on the device; the plan stays lens-free).
  int64_t target = num_sms / plan->head_groups;
  if (target < 1) target = 1;
  int64_t U = plan->total_units;
  int64_t ctas = U < target ? U : target;
  int64_t upc = ctas > 0 ? (U + ctas - 1) / ctas : 1;
  ctas = upc > 0 ? (U + upc - 1) / upc : 0;
  if (upc > INT32_MAX || ctas > INT32_MAX / 2) return DSA_ERR_UNSUPPORTED;
  plan->units_per_cta = (int32_t)upc;
  plan->ctas_per_group = (int32_t)ctas;
  // Balancing the work (live tiles plus a per-token cost) pays off when the
  // tokens have many tiles, so ragged lengths leave many dead ones, and
  // there are enough tokens to spread; elsewhere the length scan at kernel
  // start costs more latency than it saves (measured on the five configs).
  plan->balance_live = (num_tokens >= 16 && plan->tiles_per_token >= 8) ? 1 : 0;
  // An even split whose CTAs hold whole tokens (units per CTA a multiple of
  // the tiles per token) splits no token: then there is nothing to combine.
  const bool whole = !plan->balance_live && upc % plan->tiles_per_token == 0;
  plan->split_tokens = (ctas > 1 && !whole) ? (int32_t)(ctas - 1) : 0;
  // Token boundaries: T tokens over the C CTAs of a head group make about
  // T + C token segments. With fewer than 16 tiles per segment (the widths'
  // tile counts stand in for the lengths) and 64 heads per group, the
  // producer warps stage Q and issue a token's first QK (measured: config 3
  // +5 %, config 4 +1.3 %, config 5 at T = 64 +4 %; at T = 1024, 29 tiles
  // per segment, the other form is 1.5 % faster).
  plan->producer_q =
      (plan->kernel == dsa::kKernelTc && plan->heads_per_group == 64 && d_qk == 512 &&
       (int64_t)num_tokens * plan->tiles_per_token < 16 * ((int64_t)num_tokens + ctas))
          ? 1
          : 0;
  // Split tokens merged by the run kernel itself (tensor-core kernel): the
  // CTA that completes a token's units merges its parts, at most 64 of them
  // (their weights sit in a shared-memory buffer of 64 x heads-per-group
  // floats; a token spans at most min(C, tiles per token) CTAs). One CTA
  // reads every part of the token, so this pays only while tokens have few
  // parts: about C / T + 1 on average, here at most 5 (C <= 4 T). Measured
  // against the separate merge kernel: config 3 +5 %, config 4 +2 %,
  // config 5 T = 256 +2.6 %, T = 1024 +1.2 %; at T = 8 (about 10 parts) it
  // was 11 % slower and at T = 1 (33 parts) 37 % slower.
  const int64_t span = ctas < plan->tiles_per_token ? ctas : (int64_t)plan->tiles_per_token;
  plan->merge_in_run = (plan->kernel == dsa::kKernelTc && plan->split_tokens > 0 && span <= 64 &&
                        ctas <= 4 * (int64_t)num_tokens)
                           ? 1
                           : 0;
  // Workspace: status | count[HG][T] | sel[T][2] | part_lse[HG][2C][hpg] |
  //            part_sel[2C][2] | part_o[HG][2C][hpg][512] | bounds[C+1]
  //            (| stage[T][H][512] fp32, for MXFP8 output only); each run
  //            zeroes everything before sel
  const int64_t slots = 2 * ctas;
  int64_t off = kStatusBytes;
  plan->ws_count_offset = off;
  off = align_up(off + 4 * (int64_t)plan->head_groups * num_tokens, kAlignWs);
  plan->ws_sel_offset = off;
  off = align_up(off + 8 * (int64_t)num_tokens, kAlignWs);
  plan->ws_part_lse_offset = off;
  off = align_up(off + 4 * plan->head_groups * slots * plan->heads_per_group, kAlignWs);
  plan->ws_part_sel_offset = off;
  off = align_up(off + 8 * slots, kAlignWs);
  plan->ws_part_o_offset = off;
  off = align_up(off + 4 * plan->head_groups * slots * plan->heads_per_group * (int64_t)dsa::kD,
                 kAlignWs);
  plan->ws_bounds_offset = off;
  off = align_up(off + 8 * (ctas + 1), kAlignWs);
  plan->workspace_bytes = num_tokens == 0 ? 0 : off;
  // MXFP8 output: every token's fp32 output is staged [T][H][512] after it
  plan->ws_stage_offset = off;
  plan->workspace_bytes_mx =
      num_tokens == 0 ? 0 : off + 4 * (int64_t)num_tokens * num_heads * dsa::kD;
  // Test knob, read only here: a shorter budget for every bounded device wait
  // (a wait that runs out sets DSA_ERR_TIMEOUT in the status word).
  if (const char *wb = std::getenv("DSA_DECODE_WAIT_BUDGET")) {
    const long long v = std::atoll(wb);
    if (v > 0) plan->wait_budget_cycles = v;
  }
  *workspace_bytes = (size_t)plan->workspace_bytes;
  return DSA_OK;
}

dsa_status dsa_decode_run(const dsa_decode_plan_t *plan, void *workspace,
                          size_t workspace_bytes, const void *q, int64_t q_stride_t,
                          int64_t q_stride_h, const dsa_cache_desc *swa_cache,
                          const int32_t *swa_idx, int64_t swa_idx_stride,
                          const int32_t *swa_lens, const dsa_cache_desc *extra_cache,
                          const int32_t *extra_idx, int64_t extra_idx_stride,
                          const int32_t *extra_lens, const float *sink,
                          const int64_t *positions, const float *cos_sin,
                          int64_t cos_sin_rows, float scale, void *out, float *lse,
                          dsa_stream_t stream) {
  NvtxRange range("dsa_decode_run");
  if (!out) return plan_ok(plan) ? (plan->num_tokens == 0 ? DSA_OK : DSA_ERR_INVALID_ARG)
                                 : DSA_ERR_PLAN;
  return run_impl(plan, workspace, workspace_bytes, q, q_stride_t, q_stride_h, swa_cache,
                  swa_idx, swa_idx_stride, swa_lens, extra_cache, extra_idx, extra_idx_stride,
                  extra_lens, sink, positions, cos_sin, cos_sin_rows, DSA_ROPE_NEOX, scale, out,
                  nullptr, lse, stream);
}

dsa_status dsa_decode_run_v41(const dsa_decode_plan_t *plan, void *workspace,
                              size_t workspace_bytes, const void *q, int64_t q_stride_t,
                              int64_t q_stride_h, const dsa_cache_desc *swa_cache,
                              const int32_t *swa_idx, int64_t swa_idx_stride,
                              const int32_t *swa_lens, const dsa_cache_desc *extra_cache,
                              const int32_t *extra_idx, int64_t extra_idx_stride,
                              const int32_t *extra_lens, const float *sink,
                              const int64_t *positions, const float *cos_sin,
                              int64_t cos_sin_rows, int32_t rope_style, float scale,
                              void *out, const dsa_mxfp8_out *mx, float *lse,
                              dsa_stream_t stream) {
  NvtxRange range("dsa_decode_run_v41");
  return run_impl(plan, workspace, workspace_bytes, q, q_stride_t, q_stride_h, swa_cache,
                  swa_idx, swa_idx_stride, swa_lens, extra_cache, extra_idx, extra_idx_stride,
                  extra_lens, sink, positions, cos_sin, cos_sin_rows, rope_style, scale, out, mx,
                  lse, stream);
}

dsa_status dsa_decode_combine(const dsa_decode_plan_t *plan, void *workspace,
                              size_t workspace_bytes, const float *sink, void *out,
                              float *lse, dsa_stream_t stream) {
  NvtxRange range("dsa_decode_combine");
  if (!plan_ok(plan)) return DSA_ERR_PLAN;
  if (plan->num_tokens == 0 || plan->split_tokens == 0) return DSA_OK;
  if (!out) return DSA_ERR_INVALID_ARG;
  return combine_impl(plan, workspace, workspace_bytes, sink, nullptr, nullptr, 0,
                      DSA_ROPE_NEOX, out, nullptr, lse, stream);
}

dsa_status dsa_decode_combine_v41(const dsa_decode_plan_t *plan, void *workspace,
                                  size_t workspace_bytes, const float *sink,
                                  const int64_t *positions, const float *cos_sin,
                                  int64_t cos_sin_rows, int32_t rope_style, void *out,
                                  const dsa_mxfp8_out *mx, float *lse, dsa_stream_t stream) {
  NvtxRange range("dsa_decode_combine_v41");
  return combine_impl(plan, workspace, workspace_bytes, sink, positions, cos_sin, cos_sin_rows,
                      rope_style, out, mx, lse, stream);
}

dsa_status dsa_decode_selection(const dsa_decode_plan_t *plan, const void *workspace,
                                int32_t *kept, uint32_t *checksum, dsa_stream_t stream) {
  if (!plan_ok(plan)) return DSA_ERR_PLAN;
  if (plan->num_tokens == 0) return DSA_OK;
  if (!workspace || !kept || !checksum) return DSA_ERR_INVALID_ARG;
  const char *w = static_cast<const char *>(workspace) + plan->ws_sel_offset;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // sel is [T][2] (kept, checksum): two strided 2-D copies.
  cudaError_t e = cudaMemcpy2DAsync(kept, 4, w, 8, 4, plan->num_tokens,
                                    cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpy2DAsync(checksum, 4, w + 4, 8, 4, plan->num_tokens,
                          cudaMemcpyDeviceToDevice, st);
  return cuda_status(e);
}

dsa_status dsa_decode_read_status(const void *workspace, dsa_stream_t stream,
                                  int32_t *device_status) {
  if (!workspace || !device_status) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  *device_status = v;
  return DSA_OK;
}

}  // extern "C"
