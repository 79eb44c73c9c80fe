/*
 * thd_attn.h — C ABI of libthdattn.so: forward self-attention over packed
 * variable-length (THD) tensors, and the attention padding mask, on one
 * NVIDIA GB300 (sm_103a) GPU.
 *
 * Every pointer argument named "device" is a CUDA device pointer; the library
 * never dereferences it on the host and never synchronises the stream, so
 * thd_attn_fwd and thd_padding_mask are asynchronous and may be captured in a
 * CUDA graph.  `stream` is a
 * cudaStream_t passed as void* (NULL = the legacy default stream).  The caller
 * owns every buffer.  The library allocates no device memory.
 *
 * Return values are thd_status codes.  Arguments that can be checked on the
 * host are checked before anything is launched; nothing is launched when a
 * check fails.  Device metadata (cu_seqlens*, seq_is_causal) is never read on
 * the host: invalid device metadata gives unspecified output, but every
 * address the kernels form is clamped to the buffers described by the host
 * arguments, so it does not fault.
 */
#ifndef THD_ATTN_H
#define THD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  THD_OK = 0,
  THD_ERR_ARG = -1,          /* a host-checkable argument is invalid                */
  THD_ERR_UNSUPPORTED = -2,  /* valid but not supported (head_dim, dtype, heads)    */
  THD_ERR_CUDA = -3,         /* a CUDA runtime / driver call failed                  */
  THD_ERR_WORKSPACE = -4     /* workspace missing, too small or misaligned          */
} thd_status;

typedef enum { THD_BF16 = 0, THD_FP16 = 1 } thd_dtype;

/* Bits of the device status word (workspace byte offset 8, uint32). */
#define THD_STATUS_WAIT_TIMEOUT 0x1u   /* a pipeline wait gave up; output unspecified */

/*
 * thd_attn_workspace_size — bytes of device workspace thd_attn_fwd needs.
 *
 * The workspace holds the dynamic tile scheduler's work counter (uint64 at
 * byte 0) and the device status word (uint32 at byte 8, THD_STATUS_* bits).
 * thd_attn_fwd clears both on `stream` before its kernel starts, so the
 * workspace needs no initialisation, but two calls that share one workspace
 * must not overlap on the GPU.  Alignment: 16 bytes.
 */
size_t thd_attn_workspace_size(void);

/*
 * thd_attn_fwd — softmax(scale * Q K^T [+ causal mask]) V per packed sequence,
 * with a per-sequence causal/full policy, all sequences in one kernel launch.
 *
 * Sources: THD layout and cu_seqlens — "How to pad sequences that cannot be
 * evenly split in context parallelism (CP)?" (Megatron-LM issue, repro
 * script); per-sequence policy `thd_sequence_is_causal` and the padded-slot
 * arrays cu_seqlens_*_padded — "Add per-sequence causal policy to packed THD
 * attention" (TransformerEngine PR, Changes and the pad_between_seqs review
 * comment); buffers longer than batch_size + 1 — "[PyTorch] Build the
 * attention padding mask without host syncs" (Changes).
 *
 * q            device, [T, Hq, head_dim] contiguous, dtype, 16-byte aligned.
 * k, v         device, [T, Hkv, head_dim] contiguous, dtype, 16-byte aligned.
 * cu_seqlens_q, cu_seqlens_kv
 *              device int32, >= batch_size + 1 entries; entry b+1 minus entry b
 *              is sequence b's valid length.  Entries past batch_size are
 *              never read.
 * cu_seqlens_q_padded, cu_seqlens_kv_padded
 *              device int32 or NULL.  Entry b is the first row of sequence b's
 *              slot in the packed buffer; the slot's first `length` rows are
 *              valid and the rest, up to the next slot, are pad.  NULL means
 *              sequence b starts at cu_seqlens[b] (no gaps).  Entries past
 *              batch_size - 1 are never read.
 * seq_is_causal device uint8 [>= batch_size] or NULL (all full-context): the
 *              per-sequence mask type.  0 = padding (every valid key visible);
 *              2 = padding_causal_bottom_right (key j visible to query i iff
 *              j <= i + Lkv - Lq); any other value = padding_causal, top-left
 *              (j <= i), so a bool tensor works as a causal flag.  Positions
 *              count from the sequence's first token.  Mask type names: the
 *              per-sequence policy review comment of the same PR.  Rows that
 *              see no key are written as 0 with lse -inf.
 * batch_size   >= 0.  0 writes zeros to every row of `out` (and -inf to lse).
 * max_seqlen   >= 0; a hint only (the kernels read the true lengths, and any value
 *              gives results within the parity bounds).  It sizes the scheduler's
 *              claim batches and, for head_dim 64 / 128 without a window, picks the
 *              tile layout of short sequences: with 1 <= max_seqlen <= 256, runs of
 *              consecutive sequences of at most 128 rows and keys share a tile;
 *              otherwise each (sequence, head) has its own.  Calls with hints on the
 *              same side of 256 give the same bits; across it, short sequences'
 *              rows may differ in the last place.
 * softmax_scale finite, > 0.
 * out          device, [T, Hq, head_dim], dtype.  Rows of no sequence (gaps,
 *              leading and trailing pad) are written as exact zeros.
 * lse          device float32 [Hq, T] or NULL.  Natural-log log-sum-exp of the
 *              scaled logits of each valid row; -inf on pad rows.
 * total_tokens T >= 0 (rows of q/k/v/out).
 * num_heads_q, num_heads_kv  Hq >= 1, Hkv >= 1, Hq % Hkv == 0; query head h reads
 *              key/value head h / (Hq / Hkv).
 * head_dim     a multiple of 8 in [8, 128].
 * dtype        thd_dtype (bf16 or fp16); fp32 accumulation, output rounded to
 *              nearest even.
 * workspace    device, >= thd_attn_workspace_size() bytes, 16-byte aligned.
 * stream       cudaStream_t.
 *
 * Errors: THD_ERR_ARG (bad sizes, NULL required pointer, misalignment),
 * THD_ERR_UNSUPPORTED (head_dim, Hq % Hkv), THD_ERR_WORKSPACE, THD_ERR_CUDA.
 */
int thd_attn_fwd(const void* q, const void* k, const void* v,
                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                 const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                 const uint8_t* seq_is_causal,
                 int batch_size, int max_seqlen, float softmax_scale,
                 void* out, float* lse,
                 int total_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                 int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * thd_attn_fwd_window — thd_attn_fwd with a sliding window (local attention).
 *
 * Source: the window is named only as an option the per-sequence policy PR
 * rejects ("Add per-sequence causal policy to packed THD attention", Changes);
 * it is taken as a band around the diagonal of each sequence's mask type.
 * With shift = Lkv - Lq for bottom-right sequences (mask type 2) and 0
 * otherwise, key j of a sequence is visible to its query i iff it is visible
 * under the sequence's mask type and
 *     i + shift - window_left <= j <= i + shift + window_right.
 * window_left, window_right  >= -1; -1 leaves that side unbounded, so
 *              (-1, -1) is exactly thd_attn_fwd.  A causal mask type already
 *              bounds the right side at the diagonal.
 * Every other argument, the results on pad rows and rows that see no key, and
 * the errors are those of thd_attn_fwd (THD_ERR_ARG also for an extent < -1).
 * Work scales with the window: KV tiles outside every row's band of a query
 * tile are not visited.
 */
int thd_attn_fwd_window(const void* q, const void* k, const void* v,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                        const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                        const uint8_t* seq_is_causal,
                        int batch_size, int max_seqlen, float softmax_scale,
                        void* out, float* lse,
                        int total_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                        int dtype, int window_left, int window_right,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * thd_attn_bwd_workspace_size — bytes of device workspace thd_attn_bwd needs for
 * T = total_tokens rows, Hq query heads and head_dim d:
 * 256 + (Hq*T*4 rounded up to 256) + (T*Hq*d*4 rounded up to 256); 0 for invalid sizes.
 * Layout: work counter and status word as in thd_attn_workspace_size, then
 * D = rowsum(dO * O) (fp32 [Hq, T]), then the fp32 dQ accumulator [T, Hq, d].
 */
size_t thd_attn_bwd_workspace_size(int total_tokens, int num_heads_q, int head_dim);

/*
 * thd_attn_bwd — gradients dQ, dK, dV of thd_attn_fwd, for the same packed
 * batch, gaps, per-sequence mask types and grouped heads.
 *
 * Source: "Add per-sequence causal policy to packed THD attention"
 * (TransformerEngine PR, Changes and Validation: forward and Q/K/V gradient
 * parity of mixed, all-causal and all-full packed batches).  With
 * P = exp(scale q k^T - lse): dV = P^T dO; dS = P * (dO V^T - D),
 * D = rowsum(dO * O); dQ = scale dS K; dK = scale dS^T Q; dK / dV of a
 * key/value head sum over the query heads that read it.
 *
 * q, k, v, out, lse   the forward's inputs and outputs (out and lse exactly as
 *                     thd_attn_fwd returned them; lse required).
 * dout                device [T, Hq, head_dim], dtype: gradient of out.
 * dq, dk, dv          device, shapes of q, k, v, dtype, 16-byte aligned.  Rows
 *                     of no sequence, queries that see no key and keys that no
 *                     query sees get exact zeros.
 * Other arguments as thd_attn_fwd, except: head_dim 64 or 128 only; workspace
 * of at least thd_attn_bwd_workspace_size(T, Hq, head_dim) bytes, 256-byte
 * aligned, needs no initialisation and must not be shared by calls that
 * overlap on the GPU.
 * Runs three kernels on `stream` (row sums, the main pass, dQ conversion); no
 * host synchronisation.  Errors as thd_attn_fwd.
 */
int thd_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                 const void* dout,
                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                 const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                 const uint8_t* seq_is_causal,
                 int batch_size, int max_seqlen, float softmax_scale,
                 void* dq, void* dk, void* dv,
                 int total_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                 int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * thd_attn_bwd_window — thd_attn_bwd for a forward computed with
 * thd_attn_fwd_window: the same window_left / window_right (>= -1, -1 =
 * unbounded; (-1, -1) is exactly thd_attn_bwd).  Keys outside every query's
 * band get exact zero dK / dV.  Other arguments and errors as thd_attn_bwd.
 */
int thd_attn_bwd_window(const void* q, const void* k, const void* v, const void* out, const float* lse,
                        const void* dout,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                        const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                        const uint8_t* seq_is_causal,
                        int batch_size, int max_seqlen, float softmax_scale,
                        void* dq, void* dk, void* dv,
                        int total_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                        int dtype, int window_left, int window_right,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * thd_attn_fwd_noalloc — thd_attn_fwd for callers that cannot allocate device
 * memory: identical arguments minus the workspace, identical results.
 *
 * The pages have no counterpart to this entry point; it exists for the
 * library's callers.  Plugins whose host engine owns all device memory and
 * offers them no allocator, pipelines that fix their device-memory budget at
 * start-up and forbid allocation afterwards, and latency-bound loops that must
 * not risk cudaMalloc's device-wide blocking cannot provide the small
 * workspace thd_attn_fwd asks for.  Here the workspace is a fixed 256-byte
 * buffer compiled into the library (a __device__ array, one copy per GPU that
 * loads the library, kept until the process exits).  The library calls no
 * cudaMalloc/cudaFree or other allocating routine.
 *
 * - The first call on each device looks up that buffer's device address
 *   (cudaGetSymbolAddress, which may load the library's device code): make the
 *   first call on a device before any stream capture begins.
 * - Every call on a device shares the buffer.  Calls that overlap on the GPU
 *   (unordered streams) race on it and give wrong results; order them.  The
 *   buffer's counter and status word are cleared on `stream` at the start of
 *   each call; it keeps the last call's contents.
 * - THD_ERR_WORKSPACE if the library's workspace requirement ever exceeds the
 *   fixed buffer; otherwise the same status codes as thd_attn_fwd.
 * - A pipeline wait that gives up sets THD_STATUS_WAIT_TIMEOUT in the buffer's
 *   status word, exactly as in thd_attn_fwd's workspace; read it with
 *   thd_attn_noalloc_status.  The call's own return value reports only the
 *   host-side checks and the launch.
 * - The buffer's address is cached per device for the life of the process:
 *   do not keep using this entry point across cudaDeviceReset.
 */
int thd_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                         const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                         const uint8_t* seq_is_causal,
                         int batch_size, int max_seqlen, float softmax_scale,
                         void* out, float* lse,
                         int total_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                         int dtype, void* stream);

/*
 * thd_attn_noalloc_status — copies the device status word (THD_STATUS_* bits)
 * of thd_attn_fwd_noalloc's fixed buffer on the current device to *status.
 *
 * No counterpart on the pages: it completes thd_attn_fwd_noalloc, whose callers
 * hold no workspace of their own to read the status word from.  The copy is
 * queued on `stream` after the work already queued there, and the calling host
 * thread waits for it (this call synchronises `stream`), so it reports the last
 * no-allocation call on this device ordered before it.  Allocates nothing.
 * status: host pointer to one uint32.  Errors: THD_ERR_ARG (NULL status),
 * THD_ERR_CUDA.
 */
int thd_attn_noalloc_status(uint32_t* status, void* stream);

/*
 * thd_padding_mask — the boolean attention padding mask built on the device,
 * mask[b, p] = (p >= cu_seqlens[b+1] - cu_seqlens[b]) for b < batch_size,
 * p < max_seqlen (1 = padded position).
 *
 * Source: "[PyTorch] Build the attention padding mask without host syncs"
 * (TransformerEngine PR): the vectorised form (Description), the
 * [1 : batch_size + 1] slice that ignores longer buffers (Changes), and the
 * all-False row of a sequence longer than max_seqlen (Equivalence).
 *
 * cu_seqlens   device int32, >= batch_size + 1 entries (only those are read).
 * batch_size   >= 0;  max_seqlen >= 0.  Either 0: nothing is launched.
 * mask         device uint8 [batch_size * max_seqlen] (the [B, 1, 1, S] bool
 *              tensor's bytes), any alignment; every byte is written 0 or 1.
 * Errors: THD_ERR_ARG (negative sizes, NULL pointers, B*S overflow), THD_ERR_CUDA.
 */
int thd_padding_mask(const int32_t* cu_seqlens, int batch_size, int max_seqlen,
                     uint8_t* mask, void* stream);

/*
 * thd_padding_mask_cross — the cross-attention pair of padding masks: the query
 * mask from cu_seqlens_q over max_seqlen_q positions and the key/value mask from
 * cu_seqlens_kv over max_seqlen_kv positions, each exactly as thd_padding_mask.
 *
 * Source: "[PyTorch] Build the attention padding mask without host syncs"
 * (TransformerEngine PR), Equivalence (the cross-attention case: q and kv
 * lengths per sequence).
 * Arguments as thd_padding_mask; mask_q is [B*Sq] bytes, mask_kv [B*Skv] bytes.
 * batch_size 0 launches nothing.  Errors: THD_ERR_ARG, THD_ERR_CUDA.
 */
int thd_padding_mask_cross(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch_size,
                           int max_seqlen_q, int max_seqlen_kv, uint8_t* mask_q, uint8_t* mask_kv,
                           void* stream);

/*
 * thd_attn_merge — attention over the union of two disjoint key sets, from the
 * two partial results: with S = exp(lse_a) + exp(lse_b) per (row, head),
 * lse = log S and out = exp(lse_a - lse) out_a + exp(lse_b - lse) out_b.  A
 * partial whose lse is -inf saw no key and gets weight 0; if both are -inf the
 * row is 0 with lse -inf.
 *
 * Source: the context-parallel split of "How to pad sequences that cannot be
 * evenly split in context parallelism (CP)?" (Megatron-LM issue; each rank's
 * key chunk gives one partial) and the out_causal + out_non_causal sum of the
 * pad_between_seqs review comment in "Add per-sequence causal policy to packed
 * THD attention" (every row has one -inf partial there).
 *
 * out_a, out_b, out  device [T, H, head_dim] dtype, 16-byte aligned; out may be
 *                    out_a or out_b (in place).
 * lse_a, lse_b, lse  device float32 [H, T]; lse may be lse_a or lse_b.
 * total_tokens T >= 0 (0 launches nothing), num_heads H >= 1, head_dim a multiple
 * of 8 in [8, 128], dtype thd_dtype.  The merge is computed in fp32 and rounded
 * to nearest even.  Errors: THD_ERR_ARG, THD_ERR_UNSUPPORTED, THD_ERR_CUDA.
 */
int thd_attn_merge(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b,
                   void* out, float* lse, int total_tokens, int num_heads, int head_dim, int dtype,
                   void* stream);

/*
 * thd_set_wait_limit_ns — the time limit of one pipeline wait inside the
 * attention kernels (forward, windowed forward, no-allocation forward,
 * backward), for calls made after it on any host thread; returns the previous
 * limit.  0 restores the default of 2 s.
 *
 * No counterpart on the pages: it belongs to the library's failure handling.
 * Every wait of a kernel on its own pipeline (a copy landing, an MMA
 * completing, a hand-off between warps) is bounded by this limit; a wait that
 * runs out sets THD_STATUS_WAIT_TIMEOUT in the call's status word, the CTA
 * stops taking work, lets the copies and MMAs it already started finish,
 * releases its tensor memory and exits, and the call's output is unspecified.
 * No wait is expected to come near the default; a short limit makes the waits
 * run out on purpose, which is how the failure path itself is tested.
 */
uint64_t thd_set_wait_limit_ns(uint64_t ns);

/*
 * thd_set_wait_injection — test setting of the failure path: with enable != 0,
 * every CTA of the attention kernels (forward, windowed forward, no-allocation
 * forward, backward) called after it makes one wait on a barrier that nothing
 * completes before the CTA's end.  That wait runs out after the limit of
 * thd_set_wait_limit_ns whatever the timing of the rest of the pipeline, so the
 * call sets THD_STATUS_WAIT_TIMEOUT and its CTAs leave through the failure path
 * (with their copies and MMAs in flight) every time; its output is unspecified.
 * enable = 0 (the default) turns it off.  Returns the previous setting (0 or 1).
 *
 * No counterpart on the pages: it belongs to the library's failure handling and
 * exists for its tests; nothing faults, traps or hangs.
 */
int thd_set_wait_injection(int enable);

/* Human-readable name of a thd_status value (static storage). */
const char* thd_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* THD_ATTN_H */
