/*
 * libmla: the Multi-head Latent Attention (MLA) forward on one GB300 (sm_103a).
 *
 * Plain C ABI.  Tensors are caller-owned device pointers (bf16 = IEEE
 * bfloat16 stored as 16-bit words, fp32, int32) with the layouts stated per
 * call; scalar sizes are plain integers; `stream` is a cudaStream_t passed as
 * void* (NULL = the legacy default stream).  Every call is asynchronous on
 * that stream, validates its arguments on the host before launching anything,
 * and returns an mla_status.  No call allocates device memory: scratch space
 * ("workspace") is sized by the matching *_workspace_size() call and owned by
 * the caller.  No call synchronises the stream except mla_check_device_status.
 *
 * Errors: a non-MLA_OK status means nothing was launched (argument errors) or
 * a CUDA launch failed (MLA_ERR_CUDA).  mla_last_error_string() describes the
 * last failure of the calling thread.  Kernels bound every wait; a wait that
 * runs out, or an index that is out of range on the device (a page id, a
 * top-k index beyond the cache), is recorded in a status word inside the
 * workspace: mla_check_device_status() reads and clears it.
 *
 * Conventions shared by the attention calls (the passages defining them):
 *  - Scores are s = scale * (q . k) over every column of q/k; the softmax is
 *    over the visible keys; out = sum softmax(s) v; lse = max + ln(sum exp(s - max))
 *    in natural log (Huawei Ascend "RingMLAOperation", softmaxLse row:
 *    "QK^T x tor. softmax, exp, sum, and log ... in sequence").
 *  - A row with no visible key has out = 0 and lse = -inf, and merging such a
 *    row never produces NaN (NVIDIA TensorRT-LLM "mla.py", _attn_forward_gen,
 *    on 0 * NaN poisoning a combine).
 *  - A previous pair (prev_out, prev_lse) is merged by its LSE:
 *    m = max(lse_p, lse), w_p = e^(lse_p - m), w = e^(lse - m),
 *    out = (w_p out_p + w out) / (w_p + w), lse = m + ln(w_p + w)
 *    (Ascend "RingMLAOperation", prevOut / prevLse / calcType rows;
 *    TensorRT-LLM "mla.py", forward_context_with_chunked_prefill,
 *    merge_attention_for_mla).  prev_out and prev_lse are both given or both
 *    NULL (calcType FIRST_RING passes neither).  prev_lse is fp32.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* bad pointer, shape, stride, alignment or scalar */
  MLA_ERR_UNSUPPORTED = 2,  /* valid by the pages but not built (e.g. another head width) */
  MLA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  MLA_ERR_TIMEOUT = 4,      /* a kernel's bounded wait ran out (from mla_check_device_status) */
  MLA_ERR_DEVICE_RANGE = 5, /* a kernel met an out-of-range index (from mla_check_device_status) */
  MLA_ERR_WORKSPACE = 6     /* workspace NULL or smaller than *_workspace_size() */
} mla_status;

/* Library version (major * 10000 + minor * 100 + patch). */
int mla_version(void);

/* Text of the last failure on the calling thread ("" if none).  Owned by the library. */
const char* mla_last_error_string(void);

/* Static name of a status code. */
const char* mla_status_string(mla_status s);

/*
 * Reads and clears the device status word in `workspace` (any workspace that
 * a call of this library was given).  Synchronises `stream` first.  Returns
 * MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_DEVICE_RANGE; `detail` (nullable)
 * receives the raw word (wait or check site id): 0x1000 | wait site for a timeout,
 * 0x2000 | check site for an out-of-range page id or length, and, in the guarded build
 * (libmla_guard.so, compiled with MLA_GUARD), 0x3000 | site for a plain load or store of a
 * kernel that would have left its buffer (the access was skipped).
 */
mla_status mla_check_device_status(void* workspace, void* stream, uint32_t* detail);

/*
 * Bound on the spin iterations of every device wait (default 1<<25; 0 restores
 * the default).  A small value makes waits run out: tests use it to check that
 * a timeout is reported as MLA_ERR_TIMEOUT without hanging.  Process-wide.
 */
void mla_set_spin_limit(uint32_t spin_limit);

/*
 * Keys per score tile of mla_prefill (and of mla_sparse, which follows the prefill setting) and
 * of mla_decode: 128 runs the 128-key tile engine, 64 the 64-key engine.  0 restores the default of each
 * (128 for both: the faster engine for each on GB300); any other value leaves
 * the setting unchanged.  Process-wide; both engines give the same results within the
 * stated tolerances (the tests run both).
 */
void mla_set_tile_keys(int prefill_keys, int decode_keys);

/*
 * Fault injection for tests (host-side switch, process-wide): when enabled,
 * the MMA warp of every CTA launched afterwards first waits on a barrier that
 * nothing arrives on, so that wait runs out of its bound and the call reports
 * MLA_ERR_TIMEOUT through mla_check_device_status.  Off by default.
 */
void mla_debug_inject_stall(int enable);

/* ------------------------------------------------------------------------- */
/* Absorbed causal MLA prefill (one shared KV head)                          */
/* ------------------------------------------------------------------------- */
/*
 * Defined by: Tenstorrent "ttnn.transformer.ring_mla" (causal ring MLA over a
 * single KV tensor: QK^T over the full KV width, V = the first head_dim_v
 * columns, one shared KV head; is_balanced; kv_actual_isl / logical_n), and
 * TensorRT-LLM "mla.py" (forward_context_with_chunked_prefill: cached chunks
 * FULL, current chunk CAUSAL, merged by LSE).  One call is one ring step / one
 * KV chunk; a whole sequence is several calls that pass (out, lse) back as
 * (prev_out, prev_lse).
 *
 * q        bf16 [T, H, dk]; row (t, h) at q + t*q_stride_t + h*q_stride_h
 *          (element strides); the dk columns are contiguous; 16-byte aligned rows.
 * kv       bf16 [Tkv, dk]; row j at kv + j*kv_stride; kv 16-byte aligned and
 *          kv_stride*2 a multiple of 16 bytes.  Key j has global position kv_pos0 + j.
 * T, H     query tokens and query heads (H >= 1); query token t has global
 *          position q_pos0 + t.
 * Tkv      rows of kv; kv_valid (<= Tkv) rows exist (a padded chunk); -1 = Tkv.
 * dk, dv   576 and 512 (the DeepSeek latent geometry; others -> MLA_ERR_UNSUPPORTED).
 * scale    multiplies q.k (required; no default).
 * causal   1: key j is visible to token t iff kv_pos0 + j <= q_pos0 + t; 0: all valid keys.
 * prev_out bf16 [T, H, dv] contiguous, prev_lse fp32 [H, T]; both or neither.
 * out      bf16 [T, H, dv] contiguous (T * H below 2^31); may be the same buffer as prev_out.
 * lse      fp32 [H, T]; may be the same buffer as prev_lse.
 * workspace/_bytes  >= mla_prefill_workspace_size(T, H).
 */
size_t mla_prefill_workspace_size(int T, int H);
mla_status mla_prefill(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* kv, int64_t kv_stride,
                       int T, int H, int Tkv, int dk, int dv, float scale, int causal, int64_t q_pos0,
                       int64_t kv_pos0, int kv_valid, const void* prev_out, const float* prev_lse, void* out,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * A batch of sequences packed back to back (Tenstorrent "ttnn.transformer.ring_mla": batched
 * inputs with per-sequence valid lengths; TensorRT-LLM "mla.py": context attention over a batch
 * of requests).  Sequence b owns query tokens [cu_seqlens_q[b], cu_seqlens_q[b+1]) of q and key
 * rows [cu_seqlens_kv[b], cu_seqlens_kv[b+1]) of kv; with causal, its cached prefix comes first:
 * its query i sees its keys j <= kv_len - q_len + i (all of them without causal).
 * q [total_q, H, 576] with strides as in mla_prefill; kv [total_kv, 576] (row stride kv_stride);
 * out [total_q, H, 512] contiguous; lse fp32 [H, total_q]; prev_out / prev_lse (both or neither)
 * as out / lse, merged per row, and out / lse may be the same buffers.
 * cu_seqlens_q / cu_seqlens_kv: HOST int32 [batch + 1], starting at 0, non-decreasing.  A
 * sequence with no query is skipped; one with no key leaves its rows at prev (or 0 / -inf).
 * Each sequence is one launch of the prefill engine on `stream`.
 */
size_t mla_prefill_varlen_workspace_size(int total_q, int H);
mla_status mla_prefill_varlen(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* kv,
                              int64_t kv_stride, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                              int H, int dk, int dv, float scale, int causal, const void* prev_out,
                              const float* prev_lse, void* out, float* lse, void* workspace, size_t workspace_bytes,
                              void* stream);

/* ------------------------------------------------------------------------- */
/* Non-absorbed split-layout prefill (Ascend RingMLAOperation)               */
/* ------------------------------------------------------------------------- */
/*
 * Defined by: Huawei Ascend "RingMLAOperation" (AtbRingMLAGetWorkspaceSize
 * parameter table).  BSND layout, contiguous:
 *   q_nope [Nq, H, 128], q_pe [Nq, H, 64], k_nope [Nkv, Hkv, 128],
 *   k_pe [Nkv, Hkv, 64], v [Nkv, Hkv, 128]   (bf16)
 * seq_len_host: HOST int32, [batch] (q and kv lengths equal, seq_len_rows = 1)
 *   or [2, batch] (row 0 q lengths, row 1 kv lengths, seq_len_rows = 2).
 *   Sequences are packed back to back in the token dimension.  batch <= 256.
 * head_num H; kv_head_num Hkv (0 means H); H % Hkv == 0 (GQA group H / Hkv).
 * qk_scale multiplies q.k.  mask_type 0 = NO_MASK, 1 = TRIU (causal, aligned
 *   bottom-right: query i of a sequence sees keys j <= kv_len - q_len + i).
 * prev_out bf16 [Nq, H, 128] / prev_lse fp32 [H, Nq]: both or neither.
 * out bf16 [Nq, H, 128] (may alias prev_out); lse fp32 [H, Nq] (may alias prev_lse).
 * The [512, 512] mask tensor, kernelType (high precision only), inputLayout
 * (BSND only) and calcType of the page are fixed by these arguments.
 * workspace: device memory of mla_prefill_split_workspace_size bytes; besides the status
 *   word it holds the counter the kernel's CTAs claim work items from (reset on `stream`
 *   before the launch), so two calls in flight at once need two workspaces.
 */
size_t mla_prefill_split_workspace_size(int Nq, int H);
mla_status mla_prefill_split(const void* q_nope, const void* q_pe, const void* k_nope, const void* k_pe,
                             const void* v, const int32_t* seq_len_host, int seq_len_rows, int batch, int head_num,
                             int kv_head_num, float qk_scale, int mask_type, const void* prev_out,
                             const float* prev_lse, void* out, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream);

/* ------------------------------------------------------------------------- */
/* Absorbed decode over a paged latent cache, split-K + LSE reduction        */
/* ------------------------------------------------------------------------- */
/*
 * Defined by: Modular Mojo "mha_single_batch_pipelined" (token generation,
 * seqlen = 1; the key range is split across CTAs and a separate reduction
 * kernel merges the parts) and TensorRT-LLM "mla.py"
 * (forward_absorption_generation: fused q [.., 512 latent | 64 rope] against
 * the paged latent cache, one KV head).
 *
 * q           bf16 [B, H, 576] contiguous (H <= 128).
 * kv_cache    bf16 [num_pages, page_size, 576] contiguous; page_size in {16, 32, 64}
 *             or a multiple of 64; num_pages * page_size below 2^31.
 * block_table DEVICE int32 [B, max_pages]: token j of request b is row
 *             j % page_size of page block_table[b][j / page_size].
 * lens        DEVICE int32 [B]: keys of request b (0 allowed: out = 0, lse = -inf);
 *             the query sits at position lens[b] - 1 and sees all lens[b] keys.
 * num_splits  CTA pairs sharing the total key range (0 = one pair per two SMs).
 * out         bf16 [B, H, 512]; lse (nullable) fp32 [B, H].
 * Page ids outside [0, num_pages) and lens beyond max_pages * page_size are
 * reported as MLA_ERR_DEVICE_RANGE by mla_check_device_status (the rows read
 * are zero-filled instead).
 */
size_t mla_decode_workspace_size(int B, int H, int num_splits);
mla_status mla_decode(const void* q, const void* kv_cache, int64_t num_pages, int page_size,
                      const int32_t* block_table, int max_pages, const int32_t* lens, int B, int H, float scale,
                      int num_splits, void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Decode with several query tokens per request and optional attention sinks.
 *
 * Several tokens: TensorRT-LLM "mla.py" (predicted_tokens_per_seq: each request generates
 * q_per_req tokens in one step -- draft tokens of speculative / multi-token prediction).  Token i
 * of request b sits at position lens[b] - q_per_req + i and sees keys 0 .. lens[b] - q_per_req + i
 * (the cache holds all of them; causal among the request's own tokens).  A token that sees no
 * key gets out = 0, lse = -inf (or the sink's logit).
 * Sinks: Modular Mojo "mha_single_batch_pipelined" (sink, sink_weights): head h's sink logit
 * sinks[h] joins the softmax denominator as one more term with no value:
 *   out = sum_j e^{s_j} v_j / (e^{sinks[h]} + sum_j e^{s_j}),  lse = ln(e^{sinks[h]} + sum_j e^{s_j}),
 * with s_j = scale * q.k_j (the sink is in the units of the scaled scores).
 *
 * q      bf16 [B, q_per_req, H, 576] contiguous; out bf16 [B, q_per_req, H, 512];
 *        lse (nullable) fp32 [B, q_per_req, H]; sinks (nullable) DEVICE fp32 [H].
 * Other arguments as mla_decode (which is this call with q_per_req = 1 and no sinks).
 * workspace_bytes >= mla_decode_ex_workspace_size(B, q_per_req, H, num_splits).
 */
size_t mla_decode_ex_workspace_size(int B, int q_per_req, int H, int num_splits);
mla_status mla_decode_ex(const void* q, int q_per_req, const void* kv_cache, int64_t num_pages, int page_size,
                         const int32_t* block_table, int max_pages, const int32_t* lens, int B, int H, float scale,
                         const float* sinks, int num_splits, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Decode over an FP8 latent cache.  Defined by: TensorRT-LLM "mla.py" (FP8 KV cache: use_fp8_mla
 * with mla_bmm1_scale / mla_bmm2_scale, the cache's scale applied to the QK and PV products).
 * kv_cache_e4m3 holds e4m3 values (one byte each, [num_pages, page_size, 576] contiguous); every
 * value stands for e4m3_value * kv_scale (one per-tensor scale, > 0).  Arguments otherwise as
 * mla_decode_ex (q bf16 [B, q_per_req, H, 576], sinks, out, lse).  The kernel converts the cache
 * rows to f16 (exactly) on the way into shared memory, runs both products on the tensor cores with
 * f16 operands (q is rounded to f16: |q| must stay below 65504) and fp32 accumulation; the cache
 * traffic is half that of the bf16 cache.  Always runs the 128-key tile engine.
 * workspace_bytes >= mla_decode_fp8_workspace_size(B, q_per_req, H, num_splits).
 */
size_t mla_decode_fp8_workspace_size(int B, int q_per_req, int H, int num_splits);
mla_status mla_decode_fp8(const void* q, int q_per_req, const void* kv_cache_e4m3, float kv_scale, int64_t num_pages,
                          int page_size, const int32_t* block_table, int max_pages, const int32_t* lens, int B, int H,
                          float scale, const float* sinks, int num_splits, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * mla_decode without a workspace, for callers that cannot allocate device
 * memory (the pages have no counterpart of this call): plug-ins handed only
 * their input and output buffers by a framework that owns every device
 * allocation, processes that forbid device allocation after start-up, and
 * callers whose memory pool cannot grow from inside the call.  Arguments as
 * mla_decode minus the workspace.  The split-K scratch is a fixed array inside
 * this library (50,446,848 bytes, about 48.1 MiB, held by every GPU that loads the library until
 * exit); limits: B <= 4096 and (B + CTA pairs) * H <= 24576, where the pairs
 * are num_splits, or half the SM count when num_splits = 0; beyond them the
 * call returns MLA_ERR_INVALID_ARG and launches nothing.  Allocates nothing.
 * The first call on a device (with it current) looks up the array's address;
 * make it before any stream capture.  Every call shares the array: calls that
 * overlap on the GPU race.  Device-side index faults are zero-filled as in
 * mla_decode but have no workspace to be read back from.
 */
mla_status mla_decode_noalloc(const void* q, const void* kv_cache, int64_t num_pages, int page_size,
                              const int32_t* block_table, int max_pages, const int32_t* lens, int B, int H,
                              float scale, int num_splits, void* out, float* lse, void* stream);

/* ------------------------------------------------------------------------- */
/* The absorption BMMs around the latent attention                            */
/* ------------------------------------------------------------------------- */
/*
 * Defined by: TensorRT-LLM "mla.py", forward_absorption_generation (per head, q_nope times
 * k_b_proj_trans transposed gives the latent part of the fused query; the latent attention
 * output times v_b_proj transposed gives the head's output; create_weights: k_b_proj_trans
 * [num_heads, kv_lora_rank, qk_nope_head_dim], v_b_proj [num_heads, v_head_dim, kv_lora_rank]).
 * bf16 in and out, fp32 accumulation, on the tensor cores.
 *
 * mla_absorb_q: q_out[t, h, 0:512] = sum_d q_nope[t, h, d] k_b_proj_trans[h, :, d].
 *   q_nope  bf16, element (t, h, d) at q_nope + t * q_nope_stride_t + h * q_nope_stride_h + d,
 *           d < 128 contiguous (a view into the projection output is fine); strides are
 *           multiples of 8 elements, q_nope_stride_h >= 128, q_nope_stride_t >= H * q_nope_stride_h.
 *   k_b_proj_trans bf16 [H, 512, 128] contiguous.
 *   q_out   bf16 with the same kind of strides (e.g. the fused query [T, H, 576]: strides
 *           (H * 576, 576)); only columns 0..511 of each row are written.
 * mla_project_out: out[t, h, 0:128] = sum_l o_latent[t, h, l] v_b_proj[h, :, l].
 *   o_latent bf16 [T, H, 512] contiguous (the out of mla_prefill / mla_decode).
 *   v_b_proj bf16 [H, 128, 512] contiguous.  out bf16 rows of 128 with strides as above.
 * workspace: >= 256 bytes (the status word).  T = 0 launches nothing.
 */
mla_status mla_absorb_q(const void* q_nope, int64_t q_nope_stride_t, int64_t q_nope_stride_h,
                        const void* k_b_proj_trans, int T, int H, void* q_out, int64_t q_out_stride_t,
                        int64_t q_out_stride_h, void* workspace, size_t workspace_bytes, void* stream);
mla_status mla_project_out(const void* o_latent, const void* v_b_proj, int T, int H, void* out,
                           int64_t out_stride_t, int64_t out_stride_h, void* workspace, size_t workspace_bytes,
                           void* stream);

/* ------------------------------------------------------------------------- */
/* Decode step: RoPE and the paged latent-cache append                        */
/* ------------------------------------------------------------------------- */
/*
 * Defined by: TensorRT-LLM "mla.py", forward_absorption_generation (q_pe and k_pe rotated at
 * the new token's position by RotaryEmbedding(head_dim = qk_rope_head_dim, is_neox); the
 * rotated q_pe is the RoPE part of the fused query; the token's latent-cache row
 * [compressed_kv | rotated k_pe] is appended to the paged cache, as mla_rope_generation /
 * mla_rope_append_paged_kv_assign_q do inside the attention op).
 *
 * q_pe       bf16 [B, H, 64], un-rotated; c_kv bf16 [B, 512]; k_pe bf16 [B, 64], un-rotated
 *            (all contiguous, 16-byte aligned).
 * positions  DEVICE int32 [B]: the new token's index in its request = the cache row it is
 *            written to (a decode afterwards passes lens[b] = positions[b] + 1).
 * cos_sin    DEVICE fp32 [max_pos, 64]: for position p the 32 cosines, then the 32 sines, of the
 *            rotation angles (any frequency scheme of the caller's model).
 * is_neox    0: pair i is (x[2i], x[2i+1]); 1: pair i is (x[i], x[i+32]).  Pair i turns by its
 *            angle: (a, b) -> (a cos - b sin, a sin + b cos), computed in fp32, stored as bf16.
 * kv_cache / num_pages / page_size / block_table / max_pages: the paged cache of mla_decode;
 *            the row of position p is row p % page_size of page block_table[b][p / page_size].
 * q_out      bf16 [B, H, 576]: columns 512..575 receive the rotated q_pe; columns 0..511 (the
 *            absorbed latent query, see mla_absorb_q) are left as they are.
 * A position outside [0, max_pos) or beyond max_pages * page_size, or a page id outside
 * [0, num_pages), skips that request and records MLA_ERR_DEVICE_RANGE in the workspace's status
 * word (mla_check_device_status).
 */
size_t mla_rope_append_workspace_size(int B);
mla_status mla_rope_append(const void* q_pe, const void* c_kv, const void* k_pe, const int32_t* positions,
                           const float* cos_sin, int max_pos, int is_neox, void* kv_cache, int64_t num_pages,
                           int page_size, const int32_t* block_table, int max_pages, int B, int H, void* q_out,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* Top-k sparse latent + RoPE attention                                       */
/* ------------------------------------------------------------------------- */
/*
 * Defined by: AWS NKI "MLA Sparse Attention CTE Kernel API Reference"
 * (mla_sparse_attention_cte_kernel: per query, absorbed latent + RoPE
 * attention over the top-k selected cache rows; B = 1, L = 512, R = 64,
 * H <= 128, softmax_scale > 0).
 *   q_lift [B, S, H, 512], q_pe [B, S, H, 64], c_kv [B, S_kv, 512],
 *   k_pe [B, S_kv, 64] (bf16, contiguous), topk DEVICE int32 [B, S, K] (flat layout).
 * An index outside [0, S_kv) is padding: skipped.  A repeated index counts
 * once per occurrence.  out bf16 [B, S, H * 512] in natural column order
 * h * 512 + l (not the MX 4-pack order of the NKI page); lse (nullable) fp32 [B, S, H].
 * B must be 1 (as on the page); K >= 1.
 */
size_t mla_sparse_workspace_size(int S, int H);
mla_status mla_sparse(const void* q_lift, const void* q_pe, const void* c_kv, const void* k_pe, const int32_t* topk,
                      int B, int S, int S_kv, int H, int K, float softmax_scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* LSE merge of two partial results                                           */
/* ------------------------------------------------------------------------- */
/*
 * Defined by: TensorRT-LLM "mla.py" (merge_attention_for_mla in
 * forward_context_with_chunked_prefill) and Ascend "RingMLAOperation"
 * (prevOut/prevLse).  out_* bf16 [rows, H, dv] contiguous, lse_* fp32 [H, rows].
 * out/lse may alias out_a/lse_a or out_b/lse_b.  dv % 8 == 0.
 */
mla_status mla_merge_lse(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b, void* out,
                         float* lse, int64_t rows, int H, int dv, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
