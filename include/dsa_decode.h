/*
 * dsa_decode.h -- C ABI of the GB300 (sm_103a) paged sparse/sliding-window
 * MQA decode-attention library (libdsa_decode.so).
 *
 * The operation (one decode step of a DeepSeek-V4-style MQA layer): for each
 * decode token t and query head h, gather the KV rows named by two slot
 * lists -- a sliding-window list and an optional "extra" (compressed or
 * top-k) list -- from paged, quantized caches; one 512-dim row serves as both
 * key and value; compute
 *     s_j  = scale * q[t,h] . k_j
 *     lse  = log sum_j exp(s_j)                       (natural log, no sink)
 *     out  = sum_j exp(s_j) k_j / (sum_j exp(s_j) + exp(sink[h]))
 * Sources: the vLLM "swapab_decode_attn" page (SwapABDecodeKernel: __call__
 * docstring for the argument meanings, stage_inputs for slot validity and
 * paged addressing, the merge step for the sink) and FlashMLA's
 * csrc/api/sparse_decode.h page (sparse_attn_decode_interface: MQA with one
 * KV head, head dim 512, optional sink / extra cache / lengths, split-KV
 * accumulators merged by a combine kernel).
 *
 * Conventions for every entry point:
 *   - All device pointers are CUDA device (or managed) memory of the current
 *     device. The caller owns every buffer, including the workspace; the
 *     library never allocates device memory and never synchronizes, except
 *     dsa_decode_read_status, which says so.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     dsa_decode_run then dsa_decode_combine must be issued in that order on
 *     one stream, with the same plan and workspace.
 *   - Argument errors are reported before anything is launched; launch
 *     failures come back as DSA_ERR_CUDA. No entry point throws or aborts.
 *   - Optional features are switched on by non-NULL pointers: the extra list,
 *     the sink, RoPE (positions + cos_sin).
 */
#ifndef DSA_DECODE_H_
#define DSA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st *dsa_stream_t;

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = -1, /* NULL where required, bad shape, bad value     */
  DSA_ERR_UNSUPPORTED = -2, /* head count / format / width not supported     */
  DSA_ERR_ALIGNMENT = -3,   /* a pointer or stride breaks an alignment rule  */
  DSA_ERR_WORKSPACE = -4,   /* workspace NULL, too small or misaligned       */
  DSA_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed          */
  DSA_ERR_TIMEOUT = -6,     /* device status: a bounded wait gave up         */
  DSA_ERR_PLAN = -7,        /* plan not made by dsa_decode_plan / mismatched */
  DSA_ERR_BOUNDS = -8       /* device status, checking build only: an access
                               outside its extent was skipped               */
} dsa_status;

/* KV record formats (one record = one slot = one 512-dim row).
 * FP8_528  : 512 e4m3 codes, then 4 little-endian fp32 scales (one per 128
 *            dims); value = code * scale.
 * NVFP4_288: 256 bytes of e2m1 nibbles (element 2i in the low nibble of byte
 *            i), then 32 e4m3 scales (one per 16 dims); value = code * scale.
 * FP8_528_UE8M0: 512 e4m3 codes, then 16 ue8m0 scale bytes (one per 32
 *            dims); value = code * 2^(byte - 127) (the V4.1 record of the
 *            swapab page, stage_inputs fp8 branch). A scale byte of 0xFF
 *            (NaN in E8M0) gives non-finite values.
 * MODEL1_584: FlashMLA's MODEL1 record (sparse_decode.h page: bytes_per_token
 *            = 448 + 64*2 + (448/64)*1 + 1 for d_qk = d_v = 512; the page
 *            gives only the byte counts, read in the order they are summed):
 *            the e4m3 codes of dims 0..447, dims 448..511 (the RoPE part)
 *            as 64 little-endian bf16 values, 7 ue8m0 scale bytes (dim
 *            d < 448 takes byte 576 + d/64), 1 unused byte. Records are
 *            8-byte aligned within a page (584 = 8 * 73).
 * Precision of the tensor-core kernels: every row is written to an f16 tile
 * as value * 2^-e, e the exponent of the row's largest block scale (clamped
 * to [-48, 48]), and 2^e is applied again in fp32 after the products, so a
 * row's magnitude does not matter. NVFP4, FP8_528_UE8M0 and MODEL1_584
 * values are then exact (ue8m0 blocks within 2^15 of the row's largest
 * scale, and block exponents in [-63, 55]; smaller blocks are rounded,
 * relative to the row's largest, below 2^-24; MODEL1's bf16 part is exact
 * down to 2^-26 of the row's largest value, e taking that part into
 * account); FP8_528 values are code * (scale * 2^-e rounded to f16),
 * rounded to f16 (relative error <= 2^-11 for blocks within 2^14 of the
 * row's largest scale; scales up to 2^55).
 * V32_656  : FlashMLA's V3.2 record (sparse_decode.h page: bytes_per_token =
 *            512 + 64*2 + (512/128)*4 for d_qk = 576, d_v = 512; only the
 *            byte counts are given): read as the FP8_528 record followed by
 *            the key's 64 further dims as little-endian bf16 (bytes
 *            528..655). Keys have 576 dims and values are their first 512;
 *            q then has 576 dims per head. Needs a plan made with d_qk = 576
 *            (dsa_decode_plan_qk), every list in this format, and no RoPE
 *            table (q arrives as the model rotated it). Precision as FP8_528
 *            for dims 0..511; the bf16 dims are exact down to 2^-26 of the
 *            row's largest value (e takes them into account).
 * Source: the swapab page (record sizes 528 and 288, NVFP4 block of 16 with
 * e4m3 scales) with the fp32-per-128 scale layout of FlashMLA's V3.2 record
 * (sparse_decode.h, bytes_per_token = 512 + ... + (512/128)*4).            */
enum {
  DSA_REC_FP8_528 = 0,
  DSA_REC_NVFP4_288 = 1,
  DSA_REC_FP8_528_UE8M0 = 2,
  DSA_REC_MODEL1_584 = 3,
  DSA_REC_V32_656 = 4
};

/* RoPE pairings of q dims 448..511 with a table row [cos(32) | sin(32)]:
 * NEOX pairs dim 448+i with 480+i, GPTJ pairs 448+2i with 449+2i (the swapab
 * page's Q RoPE); pair i uses cos[i], sin[i]. */
enum { DSA_ROPE_NEOX = 0, DSA_ROPE_GPTJ = 1 };

/* A paged cache: base[num_pages][page_stride_bytes] bytes; the record of slot
 * s lies at base + (s / page_size) * page_stride_bytes
 *                + (s % page_size) * record_bytes.
 * base: device pointer, 16-byte aligned. page_size: power of two (>= 1).
 * page_stride_bytes: >= page_size * record_bytes and a multiple of 16 (pages
 * may lie further apart than page_size * record_bytes). Slot ids outside
 * [0, num_pages * page_size) are ignored, never dereferenced.            */
typedef struct {
  const void *base;
  int64_t num_pages;
  int64_t page_stride_bytes;
  int32_t page_size;
  int32_t format; /* DSA_REC_* */
} dsa_cache_desc;

/* Launch plan. Made by dsa_decode_plan on the host from shapes only (slot
 * lengths are not read, so planning needs no device synchronization and a
 * planned step can be captured in a CUDA graph). Plain data: copy it freely;
 * callers must not edit the fields. */
typedef struct {
  int32_t magic;           /* identifies a plan made by this library         */
  int32_t abi_version;
  int32_t num_tokens;      /* T                                              */
  int32_t num_heads;       /* H                                              */
  int32_t swa_width;       /* columns of the sliding-window slot list        */
  int32_t extra_width;     /* columns of the extra slot list (0 = none)      */
  int32_t num_sms;         /* SM count the plan was made for                 */
  int32_t head_groups;     /* CTAs that split the heads of one token         */
  int32_t heads_per_group;
  int32_t tiles_swa;       /* 128-row tiles per token in each list           */
  int32_t tiles_extra;
  int32_t tiles_per_token;
  int32_t units_per_cta;   /* units per CTA of an even split (grid sizing)   */
  int32_t ctas_per_group;  /* CTAs per head group                            */
  int32_t split_tokens;    /* upper bound on tokens split over CTAs (0: every
                              token is whole in one CTA, combine is a no-op)  */
  int32_t kernel;          /* internal kernel variant                        */
  int64_t total_units;     /* T * tiles_per_token                            */
  int64_t ws_sel_offset;   /* workspace byte offsets                         */
  int64_t ws_part_lse_offset;
  int64_t ws_part_sel_offset;
  int64_t ws_part_o_offset;
  int64_t workspace_bytes;
  int64_t ws_bounds_offset; /* int64 [ctas_per_group + 1]: CTA c owns units
                              [bounds[c], bounds[c+1]), set by the run kernel
                              (see balance_live; a tile is live when its first
                              row lies below min(len, width)) and read by the
                              combine                                       */
  int64_t balance_live;     /* 1: CTA boundaries balance live tiles (set when
                              a CTA covers >= 2 tokens on average); 0: even
                              split of the units, bounds[c] = c*units_per_cta */
  int64_t ws_stage_offset;  /* fp32 [T][H][512] staging of the MXFP8 output */
  int64_t workspace_bytes_mx; /* workspace an MXFP8-output call needs
                              (dsa_decode_run_v41 / combine_v41 with mx)     */
  int64_t wait_budget_cycles; /* SM clock cycles a device wait may take before
                              the kernel gives up (DSA_ERR_TIMEOUT); 0 = the
                              default of about 2 s. Set only from the
                              DSA_DECODE_WAIT_BUDGET environment variable at
                              planning time, so tests can make a wait run
                              out on purpose                                 */
  int64_t d_qk;             /* key / query dims the plan was made for: 512, or
                              576 (V3.2 records); 0 in a zeroed plan reads
                              as 512                                        */
  int64_t producer_q;       /* 1: on the plain tensor-core form (fp8-528 /
                              NVFP4 records, no V4.1 options) the producer
                              warps stage each token's Q and issue its first
                              QK; set for 64 heads per group when the
                              schedule gives fewer than 16 tiles per token
                              segment. Either value computes the same
                              result                                        */
  int64_t merge_in_run;     /* 1: the tensor-core run kernel merges every split
                              token itself (the CTA that completes a token's
                              units merges its parts), so dsa_decode_combine
                              launches no merge; set when tokens have few
                              parts (ctas_per_group <= 4 T) and a token
                              spans at most 64 CTAs (min(ctas_per_group,
                              tiles_per_token) <= 64)                       */
  int64_t ws_count_offset;  /* int32 [head_groups][T] units done per token,
                              zeroed by each run with the status word       */
  int64_t reserved[7];
} dsa_decode_plan_t;

/* Plan one decode call.
 * Defined by: FlashMLA's sparse_decode.h page, the scheduling metadata made
 * before the decode launch (get_decoding_sched_meta, run with num_sm_parts =
 * max(num_sms / s_q, 1) parts in get_meta): here the work of all tokens is
 * cut into (token, 128-row tile) units, spread over the SMs, and the split
 * tokens' partial buffers sized (cf. lse_accum / o_accum there).
 * num_tokens >= 0; num_heads in {16, 32, 48, 64, 96, 128}; swa_width >= 1;
 * extra_width >= 0 (0 = no extra list). num_sms: SM count to spread the
 * work over (0 = query the current device). On success fills *plan and
 * *workspace_bytes (bytes of device scratch the caller must pass to run and
 * combine; 256-byte aligned; 0 is possible only for num_tokens == 0).
 * Host-only; launches nothing. */
dsa_status dsa_decode_plan(int32_t num_tokens, int32_t num_heads, int32_t swa_width,
                           int32_t extra_width, int32_t num_sms,
                           dsa_decode_plan_t *plan, size_t *workspace_bytes);

/* Defined by: FlashMLA's sparse_decode.h page, sparse_attn_decode_interface
 * (d_qk == 576 || d_qk == 512; d_qk = 576 with d_v = 512 is its V3.2 model
 * type), with the scheduling of dsa_decode_plan.
 * As dsa_decode_plan, for key / query dims d_qk: 512 (the same plan), or
 * 576 for V3.2 records. With 576 the heads are split into
 * groups of at most 32 (a 576-dim Q tile of 64 heads and the key tile do not
 * fit in shared memory together), so num_heads must be 16, 32, 64 or 128
 * (48 and 96 give DSA_ERR_UNSUPPORTED). Other d_qk: DSA_ERR_INVALID_ARG. */
dsa_status dsa_decode_plan_qk(int32_t num_tokens, int32_t num_heads, int32_t swa_width,
                              int32_t extra_width, int32_t num_sms, int32_t d_qk,
                              dsa_decode_plan_t *plan, size_t *workspace_bytes);

/* Run the fused gather + dequant + attention kernel (argument order after the
 * plan and workspace follows the problem statement: q, sliding-window cache
 * and list, extra cache and list, sink, positions, cos_sin, scale, out, lse).
 * Defined by: the swapab page, SwapABDecodeKernel.__call__ (its docstring
 * gives the arguments: paged uint8 caches whose pages may lie further apart
 * than page * record bytes, [s_q, width] int32 slot lists with -1 invalid,
 * [s_q] int32 lengths, int64 positions, the cos/sin table, the sink) and
 * FlashMLA's sparse_decode.h page, sparse_attn_decode_interface (MQA with
 * one KV head, d_v = 512, an optional extra cache with its own indices and
 * lengths, an optional attention sink, out and lse returned).
 *
 * q          : bf16 [T, H, d_qk] (d_qk = 512, or 576 with V3.2 records),
 *              element (t, h, d) at q + t*q_stride_t + h*q_stride_h + d
 *              (strides in elements, q_stride_h >= d_qk); 16-byte aligned
 *              rows.
 * swa_cache  : required. swa_idx: int32 [T, swa_idx_stride >= swa_width]
 *              slot ids (-1 = unused). swa_lens: int32 [T]; entries at
 *              positions >= clamp(len, 0, width) are ignored.
 * extra_*    : all NULL when plan->extra_width == 0, else all required, same
 *              rules as the sliding-window list.
 * sink       : fp32 [H] natural-log logits (not multiplied by scale), or NULL.
 * positions  : int64 [T] in [0, cos_sin_rows) (a position outside the
 *              table sets the device status to DSA_ERR_INVALID_ARG and uses
 *              row 0), and cos_sin: fp32
 *              [cos_sin_rows, 64] rows [cos(32) | sin(32)], 16-byte aligned;
 *              both NULL = no RoPE. With RoPE, q dims 448..511 are rotated
 *              NeoX style (dim 448+i pairs with 480+i) before the scores.
 * scale      : softmax scale (e.g. 512^-0.5), finite.
 * out        : bf16 [T, H, 512] contiguous, 16-byte aligned.
 * lse        : fp32 [T, H] contiguous (natural-log LSE over the kept rows,
 *              without the sink; -inf when no row is kept).
 * Tokens whose work the plan splits over several CTAs get their out / lse
 * from dsa_decode_combine, which must follow on the same stream. */
dsa_status dsa_decode_run(const dsa_decode_plan_t *plan, void *workspace,
                          size_t workspace_bytes, const void *q, int64_t q_stride_t,
                          int64_t q_stride_h, const dsa_cache_desc *swa_cache,
                          const int32_t *swa_idx, int64_t swa_idx_stride,
                          const int32_t *swa_lens, const dsa_cache_desc *extra_cache,
                          const int32_t *extra_idx, int64_t extra_idx_stride,
                          const int32_t *extra_lens, const float *sink,
                          const int64_t *positions, const float *cos_sin,
                          int64_t cos_sin_rows, float scale, void *out, float *lse,
                          dsa_stream_t stream);

/* Defined by: FlashMLA's sparse_decode.h page, the combine launch after the
 * decode (run_flash_mla_combine_kernel over lse_accum / o_accum with the
 * attention sink), and the production.py page's Python KV merge
 * (O = sum_i exp(lse_i) O_i / sum_i exp(lse_i), lse = log sum_i exp(lse_i)).
 * Merge the split-KV partials left in the workspace by dsa_decode_run:
 * out = sum_i e^{lse_i} O_i / (sum_i e^{lse_i} + e^{sink}), lse = log sum_i
 * e^{lse_i}, in a fixed split order (bitwise deterministic). `sink` must be
 * the pointer given to run (or NULL). Launches nothing when the plan splits
 * no token. */
dsa_status dsa_decode_combine(const dsa_decode_plan_t *plan, void *workspace,
                              size_t workspace_bytes, const float *sink, void *out,
                              float *lse, dsa_stream_t stream);

/* MXFP8 output of the V4.1 epilogue (the swapab page's merge step: inverse
 * RoPE, MXFP8 cast, "o-fused" store). For token t, head h, dim d, with
 * G = group_size, g = h / G, chunk c = d / 32 and slot ka = c * G + h % G:
 *   code (e4m3) at  (uint8_t *)data + t*data_stride_t + g*data_stride_g
 *                   + ka*32 + d % 32;
 *   scale (ue8m0 byte, one per head and chunk) = byte ka % 4 (little-endian)
 *                   of the int32 word scale[t*scale_stride_t + g*scale_stride_g
 *                   + (ka / 4)*scale_stride_w].
 * The value stored is x * 2^(127 - E) cast to e4m3 (round to nearest even,
 * saturating), E = ceil(log2(max(amax, 1e-10) * fp32(1/448))) + 127, amax =
 * max |x| over the chunk, x the fp32 output after the inverse rotation of
 * dims >= 448 (when RoPE is on).
 * data: 4-byte aligned, data strides multiples of 4. scale: 4-byte aligned.
 * group_size >= 1 and divides num_heads. The caller owns both buffers. */
typedef struct {
  void *data;
  int32_t *scale;
  int64_t data_stride_t;   /* bytes  */
  int64_t data_stride_g;   /* bytes  */
  int64_t scale_stride_t;  /* int32 words */
  int64_t scale_stride_g;
  int64_t scale_stride_w;
  int32_t group_size;
  int32_t reserved;
} dsa_mxfp8_out;

/* Defined by: the swapab page, SwapABDecodeKernel (stage_inputs: fp8 records
 * with ue8m0 scales per 32 dims and GPT-J RoPE of Q; the merge step: inverse
 * RoPE, MXFP8 cast with ue8m0 scales per 32 dims, o-fused store).
 * dsa_decode_run with the V4.1 options (the swapab page's mega-kernel call):
 *   rope_style: DSA_ROPE_NEOX or DSA_ROPE_GPTJ (used when RoPE is on).
 *   out / mx  : exactly one non-NULL. out: bf16 [T, H, 512] as in
 *               dsa_decode_run. mx: MXFP8 output; with RoPE on, dims >= 448
 *               of the output are first rotated back (the inverse of the Q
 *               rotation, same table row); that inverse is implemented for
 *               DSA_ROPE_GPTJ only (NEOX with RoPE and mx: DSA_ERR_UNSUPPORTED).
 *               With mx the workspace must hold plan->workspace_bytes_mx
 *               bytes: run leaves each token's fp32 output in it and
 *               dsa_decode_combine_v41 writes the MXFP8 output (required).
 * Every other argument as for dsa_decode_run. Split tokens get their output
 * from dsa_decode_combine_v41 (same rope_style, positions, cos_sin, out / mx). */
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
                              dsa_stream_t stream);

/* Defined by: the swapab page's merge step (steps 8-9 of
 * SwapABDecodeKernel: fixed-order merge of the partials, sink folded once,
 * then the inverse RoPE / MXFP8 / o-fused epilogue) and FlashMLA's combine
 * launch.
 * dsa_decode_combine for dsa_decode_run_v41: the same plan, workspace, sink,
 * positions, cos_sin, rope_style and output (out or mx) as given to run.
 * With mx it merges the split tokens into the staging area and then casts
 * every token to MXFP8 (one more launch, also for plans that split nothing). */
dsa_status dsa_decode_combine_v41(const dsa_decode_plan_t *plan, void *workspace,
                                  size_t workspace_bytes, const float *sink,
                                  const int64_t *positions, const float *cos_sin,
                                  int64_t cos_sin_rows, int32_t rope_style, void *out,
                                  const dsa_mxfp8_out *mx, float *lse, dsa_stream_t stream);

/* Defined by: the swapab page, stage_inputs (a list position names a row iff
 * it lies below min(length, width) and its slot id is a cache slot; invalid
 * rows read nothing). This call exports that selection for checking; the
 * pages have no call of their own for it.
 * Row-selection record of the last run+combine on this workspace: per token
 * the number of kept rows (kept[T], int32, device) and the sum mod 2^32 over
 * kept rows of fmix32(id * 0x9E3779B1 + 2*position + list) (checksum[T],
 * uint32, device; list 0 = sliding window, 1 = extra; fmix32 = MurmurHash3's
 * 32-bit finalizer). Asynchronous copy on `stream`. */
dsa_status dsa_decode_selection(const dsa_decode_plan_t *plan, const void *workspace,
                                int32_t *kept, uint32_t *checksum, dsa_stream_t stream);

/* Defined by: the argument checks of FlashMLA's sparse_attn_decode_interface
 * (TORCH_CHECK) and the swapab page's dispatch asserts, for the conditions
 * only the device sees: the device status word of the workspace (DSA_OK;
 * DSA_ERR_INVALID_ARG when a position lies outside the cos/sin table;
 * DSA_ERR_TIMEOUT when a bounded device wait gave up). SYNCHRONIZES `stream`
 * to read it. */
dsa_status dsa_decode_read_status(const void *workspace, dsa_stream_t stream,
                                  int32_t *device_status);

/* Bytes of the library's own device scratch used by dsa_decode_run_noalloc
 * (one array per device, 48 MiB). A plan for up to 152 SMs needs about
 * 40 MB plus 8 bytes per token, so every plan of up to ~1M tokens on a
 * GB300 fits. */
#define DSA_NOALLOC_MAX_WORKSPACE (48u * 1024u * 1024u)

/* dsa_decode_run followed by dsa_decode_combine, with the library's own
 * file-scope device array (DSA_NOALLOC_MAX_WORKSPACE bytes) as the
 * workspace. The pages that define the method have no counterpart of this
 * call. It serves callers that cannot provide a workspace: a plain C host
 * program without a device allocator of its own, or a runtime that has given
 * all free device memory to its KV-cache pool. A cudaMalloc inside the call
 * would also synchronize the device. The call allocates nothing.
 *   plan: from dsa_decode_plan; a plan whose workspace_bytes exceeds
 *         DSA_NOALLOC_MAX_WORKSPACE is refused with DSA_ERR_WORKSPACE
 *         before any CUDA call.
 *   q ... lse, stream: as for dsa_decode_run; out and lse receive the final
 *         (combined) result.
 *   device_status: optional int32 device pointer (4-byte aligned). When
 *         non-NULL, it receives an asynchronous copy of the device status
 *         word (DSA_OK, or what the kernels recorded, as
 *         dsa_decode_read_status reports it); DSA_OK for a plan of 0 tokens.
 *         Each call starts from a cleared status word.
 * Set-up: the first call on each device, with that device current, looks
 * the array up (cudaGetSymbolAddress, which may load the module); make that
 * first call before any stream capture. The array is shared: calls that
 * overlap in time on one device (other streams or host threads) race on it
 * and must be serialized by the caller. */
dsa_status dsa_decode_run_noalloc(const dsa_decode_plan_t *plan, const void *q,
                                  int64_t q_stride_t, int64_t q_stride_h,
                                  const dsa_cache_desc *swa_cache, const int32_t *swa_idx,
                                  int64_t swa_idx_stride, const int32_t *swa_lens,
                                  const dsa_cache_desc *extra_cache, const int32_t *extra_idx,
                                  int64_t extra_idx_stride, const int32_t *extra_lens,
                                  const float *sink, const int64_t *positions,
                                  const float *cos_sin, int64_t cos_sin_rows, float scale,
                                  void *out, float *lse, int32_t *device_status,
                                  dsa_stream_t stream);

/* Static description of a status code (no counterpart on the pages). */
const char *dsa_decode_status_string(dsa_status s);

/* ABI version of this header (bumped on any layout change; no counterpart
 * on the pages). */
int32_t dsa_decode_abi_version(void);

#define DSA_DECODE_ABI_VERSION 3

#ifdef __cplusplus
}
#endif
#endif /* DSA_DECODE_H_ */
