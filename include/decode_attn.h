/*
 * decode_attn: decode-step attention over a KV cache, GB300 (sm_103a).
 *
 * C ABI of libdecode_attn.so.  Every entry point takes plain pointers and
 * sizes.  Device pointers are caller-owned CUDA device memory on the current
 * device; the library never frees them, never synchronises, and launches all
 * work asynchronously on the given stream, so buffers must stay alive until
 * that stream has consumed them.  Every call returns a da_status; when an
 * argument check fails nothing is launched and no memory is touched.
 *
 * What is computed ("MoA-Structured Decode Attention", arXiv 2607.19456):
 *   for every sequence b and query head h, with kv = h / (h_q / h_kv)
 *   (GQA/MQA psi-selection, introduction item 4) and n = seq_lens[b]:
 *     Step I   (section 2, eq. 1)  s[l]  = scale * sum_j q[b,h,j] * K[b,kv,l,j],  l < n
 *     Step II  (section 2, eq. 2)  a[l]  = exp(s[l] - max s) / sum_l' exp(s[l'] - max s)
 *     Step III (section 2, eq. 3)  out[b,h,d] = sum_l a[l] * V[b,kv,l,d]
 *   Tensors are row-major (gamma offsets of section 3):
 *     q   [B, h_q, d_k]            dtype
 *     K   [B, h_kv, n_max, d_k]    dtype   (row l of head (b, kv) at ((b*h_kv+kv)*n_max+l)*d_k)
 *     V   [B, h_kv, n_max, d_v]    dtype
 *     out [B, h_q, d_v]            float32, or bfloat16 when dtype carries DA_OUT_BF16
 *   Rows at or beyond seq_lens[b] are never used: they may hold anything,
 *   including NaN.  A sequence with seq_lens[b] == 0 yields out = 0.
 *
 * The softmax is evaluated as a split-KV flash decode: the rows of each
 * sequence are cut into ranges of `chunk` rows, each (sequence, kv head,
 * range) produces a normalised partial output and its log-sum-exp, and a
 * combine kernel merges the ranges of every sequence that has more than one.
 * The result equals the definition above up to float rounding (fp32
 * accumulation).
 */
#ifndef DECODE_ATTN_H_
#define DECODE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DA_API __attribute__((visibility("default")))
#else
#define DA_API
#endif

/*
 * Element type of q, K, V (and of the rows appended by kv_append).  DA_INT8
 * and DA_FP8_E4M3 are 8-bit caches (the *_q8 entry points only): K and V
 * hold one-byte codes, each cached row has one float32 scale, q is bf16.
 */
typedef enum {
  DA_FP32 = 0,
  DA_BF16 = 1,
  DA_INT8 = 2,
  DA_FP8_E4M3 = 3
} da_dtype;

typedef enum {
  DA_OK = 0,
  DA_ERR_NULL = -1,        /* a required pointer is NULL */
  DA_ERR_SHAPE = -2,       /* a size is out of range or inconsistent */
  DA_ERR_DTYPE = -3,       /* unknown dtype */
  DA_ERR_ALIGN = -4,       /* a device pointer is not 16-byte aligned */
  DA_ERR_WORKSPACE = -5,   /* workspace missing or smaller than required */
  DA_ERR_CUDA = -6,        /* a CUDA runtime/driver call failed */
  DA_ERR_DEVICE = -7,      /* the current device is not sm_103 (GB300) */
  DA_ERR_UNSUPPORTED = -8  /* valid request this build has no kernel for */
} da_status;

/*
 * Flag OR-ed into the dtype argument of the decode entry points: `out` is
 * bfloat16 (round to nearest even of the fp32 result) instead of float32.
 * Split partials and the combine stay in float32; the result is rounded once.
 */
#define DA_OUT_BF16 0x100

/* Bits the kernels OR into the optional device error word. */
#define DA_DEVERR_SEQ_LEN 1 /* some seq_lens[b] outside [0, n_max]: clamped into range */
#define DA_DEVERR_POS 2     /* some kv_append pos[b] outside [0, n_max): that row not written */
#define DA_DEVERR_TIMEOUT 4 /* a pipeline wait exceeded its time limit: outputs invalid */
#define DA_DEVERR_BOUNDS 8  /* bounds-checked test builds only: an index fell outside its
                               buffer and that access was skipped; outputs invalid */

/*
 * Supported sizes: d_k == d_v in {64, 128} for every cache type, and for
 * bf16 caches also d_k == d_v == 256 and d_k = 192 with d_v = 128 (other
 * pairs return DA_ERR_UNSUPPORTED); any B, h_kv >= 1 and
 * h_q a multiple of h_kv; 1 <= n_max <= 2^30; B * h_kv * n_max rows must fit
 * in 2^31 - 1 for the tensor maps.  Alignment: q, K, V, out, k_new, v_new
 * must be 16-byte aligned.
 */

/*
 * Upper bound on the splits per sequence that decode_attn_ex may use for a
 * request (the workspace is sized for it).  With num_splits > 0 the split
 * length is the whole number of pipeline stages closest to n_max / num_splits,
 * so the bound is close to num_splits; with num_splits == 0 the kernels pick
 * the split length on the device from the actual seq_lens, never shorter than
 * this bound implies.  Returns a value >= 1, or a negative da_status.
 */
DA_API int decode_attn_resolve_splits(int B, int h_q, int h_kv, int d_k, int d_v, int n_max,
                                      int dtype, int num_splits);

/*
 * Bytes of device workspace decode_attn_ex needs for this request: a 256-byte
 * header, the per-split partial outputs and log-sum-exps (float32) of at
 * most 512 sequences (larger batches run as several launches that reuse
 * it, one after the other on the stream) and 16 KB in which each CTA leaves
 * the position of its first tiles for the next call on the same workspace
 * (read back as an L2 prefetch hint: any content is safe).  0 when the
 * request can only use one split.  Returns 0 and sets *status (when non-NULL) to a
 * negative da_status if the arguments are invalid.
 */
DA_API size_t decode_attn_workspace_bytes(int B, int h_q, int h_kv, int d_k, int d_v, int n_max,
                                          int dtype, int num_splits, int* status);

/*
 * Decode attention with a caller-provided workspace.
 *   q, K, V, out : device pointers, layouts above.
 *   seq_lens     : device int32 [B]; 0 <= seq_lens[b] <= n_max.  Values out
 *                  of range are clamped and flagged in *dev_error.
 *   scale        : multiplies q.K (typically 1/sqrt(d_k)).
 *   num_splits   : splits per (b, kv head); 0 = library's choice (equal
 *                  splits whose length the kernels pick from the lengths,
 *                  one split per unit, or balanced pieces when one split per
 *                  unit would leave more than a tenth of the grid's rounds
 *                  idle and each CTA's share is at least 8 tiles); -1 =
 *                  balanced: the rows of all (sequence, kv head) units, unit
 *                  after unit, are cut into one equal piece per SM (at tile
 *                  boundaries), for batches whose lengths differ widely (the
 *                  workspace then holds up to one partial per SM per query
 *                  head; when that exceeds 256 MiB, or the rows of a launch
 *                  slice exceed 2^31, the library's choice applies).
 *   workspace    : device memory of at least
 *                  decode_attn_workspace_bytes(...) bytes, 16-byte aligned;
 *                  may be NULL when that is 0.  Its contents need no
 *                  initialisation and are scratch after the call.  Calls
 *                  whose kernels may overlap on the GPU need separate
 *                  workspaces.
 *   dev_error    : nullable device int32; kernels OR DA_DEVERR_* bits into it
 *                  (it is never cleared by the library).
 *   stream       : CUDA stream for every launch.
 * Launches, per slice of at most 512 sequences, one split kernel and, when
 * more than one split may be used, one combine kernel (programmatic
 * dependent launch: it starts while the split kernel drains).
 */
DA_API int decode_attn_ex(const void* q, const void* K, const void* V, const int32_t* seq_lens,
                          void* out, int B, int h_q, int h_kv, int d_k, int d_v, int n_max,
                          float scale, int dtype, int num_splits, void* workspace,
                          size_t workspace_bytes, int32_t* dev_error, cudaStream_t stream);

/*
 * One decode step with the KV-cache append fused in ("MoA-Structured Decode
 * Attention", introduction item 3 followed by section 2): for every b with
 * 0 <= seq_lens[b] < n_max, row seq_lens[b] of every kv head of K and V
 * receives k_new[b, h, :] / v_new[b, h, :] (an exact copy of the bits, as
 * kv_append does) and the decode runs over seq_lens[b] + 1 rows, the new row
 * included, all in the same launch.  A sequence whose seq_lens[b] is outside
 * [0, n_max) gets no new row (DA_DEVERR_POS) and is decoded over its clamped
 * length.
 *   k_new [B, h_kv, d_k], v_new [B, h_kv, d_v] : device, dtype, 16-byte aligned
 *   seq_lens      : device int32 [B], the lengths before the append (read only)
 *   seq_lens_out  : nullable device int32 [B]; receives the lengths after the
 *                   append.  Must not be seq_lens itself.
 *   other arguments, workspace and errors: as decode_attn_ex (the workspace
 *   size is decode_attn_workspace_bytes of the same request).
 */
DA_API int decode_attn_append(const void* q, const void* k_new, const void* v_new, void* K, void* V,
                              const int32_t* seq_lens, int32_t* seq_lens_out, void* out, int B,
                              int h_q, int h_kv, int d_k, int d_v, int n_max, float scale,
                              int dtype, int num_splits, void* workspace, size_t workspace_bytes,
                              int32_t* dev_error, cudaStream_t stream);

/*
 * Decode attention with a library-owned workspace: the same computation as
 * decode_attn_ex with num_splits = 0 (library's choice).  The workspace is
 * cached per device and grown with cudaMalloc when a request needs more (a
 * growth waits for the device to go idle before freeing the old buffer), so
 * the first call of a given size must not happen during stream capture.
 * Concurrent calls on different streams of one device share that workspace
 * and must be serialised by the caller; use decode_attn_ex otherwise.
 */
DA_API int decode_attn(const void* q, const void* K, const void* V, const int32_t* seq_lens,
                       void* out, int B, int h_q, int h_kv, int d_k, int d_v, int n_max,
                       float scale, int dtype, cudaStream_t stream);

/*
 * Decode attention that allocates nothing (the pages have no counterpart:
 * this is a deployment variant of decode_attn_ex).
 *
 * For callers that cannot call cudaMalloc: a serving loop where an
 * allocation would synchronise the device and stall other streams, code
 * whose device memory is all owned and accounted by another allocator, or a
 * host runtime with no device allocator at all.  The split partials go to a
 * scratch buffer of DA_NOALLOC_SCRATCH_BYTES that the library itself holds
 * as a file-scope device array; every GPU that loads the library keeps it
 * until the process exits.  Arguments and results are those of
 * decode_attn_ex; the caller still provides q, K, V, seq_lens and out.
 *
 * Returns DA_ERR_WORKSPACE when the request needs more scratch than
 * DA_NOALLOC_SCRATCH_BYTES (see decode_attn_workspace_bytes; fewer splits
 * need less).  Balanced pieces (num_splits = -1) keep up to one partial per
 * SM per query head, which exceeds the buffer for all but small batches
 * (B = 16, h_q = 32, d_v = 128 already needs ~39 MB): such requests are
 * rejected, not served with another split choice.  When the library's own
 * choice (num_splits = 0) is balanced pieces that do not fit, the call takes
 * one split per sequence instead (as num_splits = 1 would).  Calls no cudaMalloc,
 * cudaFree or other allocating routine.  The first call on a device looks up
 * the buffer's device address with that device current and caches it with
 * the id of the device's current context (a call after cudaDeviceReset looks
 * it up again); make that first call before any stream capture.  All calls share the one buffer, which keeps the last call's
 * contents (nothing in it needs to start at zero): calls whose kernels may
 * overlap on the GPU (different streams, or several host threads) race on it
 * and must be serialised by the caller.
 */
#define DA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

DA_API int decode_attn_noalloc(const void* q, const void* K, const void* V, const int32_t* seq_lens,
                               void* out, int B, int h_q, int h_kv, int d_k, int d_v, int n_max,
                               float scale, int dtype, int num_splits, int32_t* dev_error,
                               cudaStream_t stream);

/*
 * Sequence-sharded decode, the per-shard half.  When the cached rows of a
 * sequence are spread over several GPUs (or several row ranges of one
 * cache), each holder decodes its own rows and the exact softmax over all of
 * them is recovered by a log-sum-exp merge of the per-holder results ("Phase
 * 3, Section 6: StoryLM-0 head-parallel attention" shards attention across
 * devices and gathers the shards; split by rows, the gather is this merge).
 * For every b and query head h, with n = seq_lens[b] and the rows
 * R_b = [min(row_begin, n), min(row_end, n)):
 *   o[b,h,:]  = sum_{l in R_b} a_l V[b,kv,l,:], a the softmax of Steps I-II
 *               of decode_attn_ex taken over R_b only (normalised);
 *   lse[b,h]  = log sum_{l in R_b} exp(s_l), natural log, s_l the scaled
 *               scores of Step I;
 *   an empty R_b gives o = 0 and lse = -inf.
 *   o   : device float32 [B, h_q, d_v]      lse : device float32 [B, h_q]
 *   row_begin, row_end : 0 <= row_begin <= row_end; rows past n are ignored.
 * dtype is DA_FP32 or DA_BF16 (no DA_OUT_BF16: partials stay float32);
 * other arguments, workspace and errors as decode_attn_ex (the workspace size
 * is decode_attn_workspace_bytes of the same request).
 */
DA_API int decode_attn_partial(const void* q, const void* K, const void* V,
                               const int32_t* seq_lens, int row_begin, int row_end, float* o,
                               float* lse, int B, int h_q, int h_kv, int d_k, int d_v, int n_max,
                               float scale, int dtype, int num_splits, void* workspace,
                               size_t workspace_bytes, int32_t* dev_error, cudaStream_t stream);

/*
 * Sequence-sharded decode, the merge half: combines S partial results over
 * disjoint row sets, as produced by decode_attn_partial and gathered by the
 * caller into this GPU's own memory (a partial is never read from a peer):
 *   L = max_s lse_s;  out = sum_s e^(lse_s - L) o_s / sum_s e^(lse_s - L);
 *   lse_out = L + log(sum_s e^(lse_s - L))      (-inf and out = 0 when every
 *   part is empty), which equals the decode over the union of the rows.
 *   o_parts   : device float32 [S, B, h_q, d_v], 16-byte aligned
 *   lse_parts : device float32 [S, B, h_q], natural log
 *   out       : device [B, h_q, d_v], float32, or bf16 when out_dtype is
 *               DA_FP32 | DA_OUT_BF16; 16-byte aligned
 *   lse_out   : nullable device float32 [B, h_q]
 *   d_v in {64, 128, 256}; S >= 0 (S = 0 gives out = 0, lse_out = -inf, and
 *   o_parts / lse_parts may then be NULL).
 * One kernel launch on `stream`.
 */
DA_API int decode_attn_combine(const float* o_parts, const float* lse_parts, int S, void* out,
                               float* lse_out, int B, int h_q, int d_v, int out_dtype,
                               cudaStream_t stream);

/*
 * KV-cache accumulation ("MoA-Structured Decode Attention", introduction
 * item 3, with the gamma offsets of section 3): for every b < B, h < h_kv
 *   K[b, h, pos[b], :] = k_new[b, h, :]     (d_k elements)
 *   V[b, h, pos[b], :] = v_new[b, h, :]     (d_v elements)
 * as an exact copy of the bits.
 *   k_new [B, h_kv, d_k], v_new [B, h_kv, d_v] : device, dtype
 *   K, V  : the caches, written in place
 *   pos   : device int32 [B], the row to write (normally the current
 *           seq_lens[b]); a pos outside [0, n_max) writes nothing for that
 *           sequence and sets DA_DEVERR_POS in *dev_error.
 * Does not change seq_lens: the caller advances it.
 */
DA_API int kv_append(const void* k_new, const void* v_new, void* K, void* V, const int32_t* pos,
                     int B, int h_kv, int d_k, int d_v, int n_max, int dtype,
                     int32_t* dev_error, cudaStream_t stream);

/*
 * 8-bit KV caches ("Attention over the KV cache in the decode step" notes
 * that an int8 or fp8 cache halves the bytes per cached row and doubles the
 * arithmetic intensity; the pages fix no format, so this one is the
 * library's).  A cached row of K (or V) is d one-byte codes c[j] plus one
 * float32 scale s, and stands for s * value(c[j]):
 *   DA_INT8      value = the two's-complement integer (-128 .. 127)
 *   DA_FP8_E4M3  value = the fp8 e4m3 number (bias 7, 3 mantissa bits,
 *                subnormals below 2^-6, S.1111.111 the only NaN, max 448)
 * Layouts (row-major, device):
 *   K, V            [B, h_kv, n_max, d]  codes (1 byte each)
 *   k_scale, v_scale [B, h_kv, n_max]    float32, one per cached row,
 *                                        16-byte aligned
 *   q               [B, h_q, d]          bfloat16
 *   out             as decode_attn_ex (float32, or bf16 with DA_OUT_BF16)
 * The decode computes Steps I-III of decode_attn_ex on the values the codes
 * and scales stand for; fp16 tensor cores see the codes' exact values, the
 * scales are applied in float32.  Row scales must be finite and below 65504
 * in magnitude; rows at or beyond seq_lens[b] may hold anything.  Extra
 * requirements: n_max a multiple of 4; d_k == d_v in {64, 128}.
 */

/* Decode over an 8-bit cache; arguments as decode_attn_ex plus the row
 * scales.  dtype is DA_INT8 or DA_FP8_E4M3 (| DA_OUT_BF16); the workspace
 * size is decode_attn_workspace_bytes of the same dtype. */
DA_API int decode_attn_q8_ex(const void* q, const void* K, const void* V, const float* k_scale,
                             const float* v_scale, const int32_t* seq_lens, void* out, int B,
                             int h_q, int h_kv, int d_k, int d_v, int n_max, float scale,
                             int dtype, int num_splits, void* workspace, size_t workspace_bytes,
                             int32_t* dev_error, cudaStream_t stream);

/* decode_attn_append for an 8-bit cache: the new rows arrive as codes
 * k_new/v_new [B, h_kv, d] (1 byte each, 16-byte aligned) with their scales
 * k_new_scale/v_new_scale [B, h_kv] (float32); codes and scale are copied
 * into row seq_lens[b] of the caches and take part in the same decode. */
DA_API int decode_attn_q8_append(const void* q, const void* k_new, const void* v_new,
                                 const float* k_new_scale, const float* v_new_scale, void* K,
                                 void* V, float* k_scale, float* v_scale, const int32_t* seq_lens,
                                 int32_t* seq_lens_out, void* out, int B, int h_q, int h_kv,
                                 int d_k, int d_v, int n_max, float scale, int dtype,
                                 int num_splits, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_error, cudaStream_t stream);

/* kv_append for an 8-bit cache: row pos[b] of every kv head receives the
 * code rows k_new/v_new [B, h_kv, d] and the scales k_new_scale/v_new_scale
 * [B, h_kv], bit for bit; errors as kv_append. */
DA_API int kv_append_q8(const void* k_new, const void* v_new, const float* k_new_scale,
                        const float* v_new_scale, void* K, void* V, float* k_scale,
                        float* v_scale, const int32_t* pos, int B, int h_kv, int d_k, int d_v,
                        int n_max, int dtype, int32_t* dev_error, cudaStream_t stream);

/* Quantize rows x [rows, d] (x_dtype DA_FP32 or DA_BF16, device) into codes
 * [rows, d] (code_dtype DA_INT8 or DA_FP8_E4M3) and scales [rows] (float32):
 * a = max_j |x[j]|, s = a / Q (Q = 127 or 448, float32 division),
 * code[j] = round-to-nearest-even(x[j] / s) clamped to [-Q, Q], all codes 0
 * when s = 0.  x must be finite; d a multiple of 32, at most 256. */
DA_API int kv_quantize(const void* x, int x_dtype, void* codes, float* scales, long long rows,
                       int d, int code_dtype, cudaStream_t stream);

/* Static, human-readable name of a da_status. */
DA_API const char* decode_attn_status_string(int status);

/* Text of the last CUDA error a call on this host thread ran into ("" if none). */
DA_API const char* decode_attn_last_cuda_error(void);

/* Number of kernels this library has launched in this process (all devices). */
DA_API uint64_t decode_attn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H_ */
