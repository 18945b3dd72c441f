/*
 * gqa_attn.h -- C ABI of libgqa_attn.so: fused causal grouped-query attention,
 * forward and backward, for NVIDIA GB300 (sm_103a).
 *
 * What the library computes
 *   Attention as the tang page states it ("How tang works", section 3,
 *   "Optimizations are derived, not written", equations (5)-(6)): the row
 *   softmax of scale * Q K^T over the visible keys, applied to V, evaluated
 *   as the streaming reduction whose three running values (row max m, sum l,
 *   accumulator) form an associative combine, so that no S x S score matrix
 *   is ever written. Grouped-query heads as in the RustingBrain docs ("GQA
 *   12/4 heads", ".heads(8, 2, 64)"): Hq query heads share Hkv key/value
 *   heads, query head h reads KV head h / (Hq / Hkv). The backward is the
 *   gradient of sum(O * dO), itself a comprehension with no S x S
 *   intermediates (aiinsiders.net, "A compiler that derives GPU kernels
 *   matches hand-tuned code"), with f32 accumulation throughout (the same
 *   article reports a bf16-accumulating fused backward missing the f32
 *   tolerance).
 *
 * Layout (every tensor dense, row-major, "BHSD"):
 *   q, o, dO, dq : bf16 [B, Hq,  S, D]
 *   k, v, dk, dv : bf16 [B, Hkv, S, D]
 *   lse          : f32  [B, Hq,  S]      natural-log log-sum-exp of the scaled scores
 * Every pointer is a DEVICE pointer, 16-byte aligned (TMA requirement).
 * Causal: key j is visible to query i iff j <= i (queries and keys share the
 * length S). causal = 0 makes every key visible.
 * Supported: D in {64, 128}; any S >= 1; B, Hq, Hkv >= 1 with Hq % Hkv == 0;
 * B * Hq * ceil(S / 128) * 128 below 2^31.
 *
 * Ownership: the caller allocates and owns every buffer (device memory and
 * the stream). The library never allocates or frees device memory and never
 * synchronises the stream, except gqa_attn_get_error(). All work is enqueued
 * on `stream` (a cudaStream_t; NULL means the legacy default stream) and runs
 * asynchronously with respect to the host.
 *
 * Errors: every entry point returns GQA_OK (0) or a negative code. Invalid
 * arguments are rejected on the host before anything is enqueued. A CUDA
 * launch failure returns GQA_ERR_CUDA (the CUDA error code is kept, per host
 * thread, for gqa_attn_last_cuda_error()). A device-side wait that exceeds
 * its time limit makes the kernel give up cleanly and sets a device status
 * bit that gqa_attn_get_error() reports as GQA_ERR_TIMEOUT. There is no CPU
 * fallback of any kind: a failure is an error code.
 *
 * Thread safety: entry points may be called concurrently from several host
 * threads. Device-side errors are kept per stream (see gqa_attn_get_error).
 *
 * Profiling: every entry point and every kernel launch is bracketed by an
 * NVTX range named after it (a no-op unless a profiling tool is attached).
 *
 * The self-test and tracing hooks used by this library's own tests and
 * benchmark are declared in gqa_attn_testing.h; they are not part of this
 * stable interface.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_OK 0
#define GQA_ERR_INVALID_ARG (-1)         /* null/misaligned pointer, bad size, Hq % Hkv != 0, scale not finite */
#define GQA_ERR_UNSUPPORTED (-2)         /* D not in {64, 128}, sizes beyond the index range */
#define GQA_ERR_WORKSPACE_TOO_SMALL (-3) /* backward workspace smaller than gqa_attn_bwd_workspace_size() */
#define GQA_ERR_CUDA (-4)                /* a CUDA runtime/driver call failed; see gqa_attn_last_cuda_error() */
#define GQA_ERR_TIMEOUT (-5)             /* a device-side wait gave up (reported by gqa_attn_get_error) */
#define GQA_ERR_INTERNAL (-6)            /* a kernel's own layout check failed and it did no work (gqa_attn_get_error) */
#define GQA_ERR_BOUNDS (-7)              /* debug build only: a computed coordinate fell outside its tensor (gqa_attn_get_error) */

/* Device status words per device: one for each of the first GQA_STATUS_STREAMS - 1 streams that
 * call into the library on that device; any further streams share one word. */
#define GQA_STATUS_STREAMS 64

/*
 * Forward: O = softmax(scale * Q K^T + causal mask) V and LSE per query row.
 *   q [B,Hq,S,D], k, v [B,Hkv,S,D] (inputs, bf16, device)
 *   o [B,Hq,S,D] (output, bf16, device), lse [B,Hq,S] (output, f32, device;
 *   lse = ln sum_j exp(scale * q_i . k_j) over the visible keys)
 *   scale: multiplies the scores (usually 1/sqrt(D)); must be finite and >= 0.
 * Passage: tang, "How tang works" section 3, equations (5)-(6) (attention as
 * written vs. the derived streaming reduction: same answer, no score matrix).
 */
int gqa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int S,
                 int D, int causal, float scale, void* stream);

/*
 * Forward over a key/value cache: Sq <= Sk query rows against Sk keys, query r
 * at absolute position Sk - Sq + r (causal: sees keys j <= Sk - Sq + r, the
 * bottom-right alignment; Sq = Sk is gqa_attn_fwd). Prefill of Sq new tokens
 * over a cache, on the tensor cores (gqa_attn_decode_fwd serves Sq with at
 * most 16 rows per KV head, split over key chunks).
 *   q, o [B,Hq,Sq,D], k, v [B,Hkv,Sk,D] (bf16, device), lse [B,Hq,Sq] (f32).
 * Errors as gqa_attn_fwd; GQA_ERR_INVALID_ARG if Sq < 1 or Sq > Sk.
 * Passage: RustingBrain docs, "Training infrastructure" (KV-cached decoding);
 * tang page, "An LLM" (prefill 512).
 */
int gqa_attn_fwd_cached(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Sq, int Sk, int D, int causal, float scale, void* stream);

/*
 * Forward over a key/value cache (as gqa_attn_fwd_cached; Sq = Sk is the training forward) that
 * splits the key range of small grids across CTAs. When the grid of query-tile pairs is small (a
 * prefill of a few hundred tokens over a long cache, short sequences), the key tiles of the longest
 * pairs are cut into contiguous parts, one CTA each, which leave their running states (m, l, O) in
 * the workspace; a second kernel on the same stream merges them by the associative combine in part
 * order: the result equals the unsplit forward's up to f32 rounding and is the same on every call.
 * Larger grids run the unsplit forward (one kernel).
 *   workspace: device memory of gqa_attn_fwd_splitkv_workspace_size() bytes (the same sizes),
 *   256-byte aligned, owned by the caller; its contents need no initialisation and are scratch
 *   until the call's kernels complete. A size of 0 means no split for these sizes: workspace may
 *   then be NULL (also accepted for other sizes: the call then runs unsplit).
 * Errors as gqa_attn_fwd_cached; GQA_ERR_WORKSPACE_TOO_SMALL for a smaller workspace.
 * Passage: tang page, "How tang works" section 3 (the combine is associative, so the key range
 * splits and the parts recombine); tang page, "An LLM" (prefill 512).
 */
size_t gqa_attn_fwd_splitkv_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D);
int gqa_attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                         float scale, void* stream);

/*
 * Forward over a packed batch of variable-length sequences: the nseq sequences
 * lie end to end along the row axis, sequence i owning query rows
 * cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1 and key/value rows cu_seqlens_k[i] ..
 * cu_seqlens_k[i+1]-1. A query attends only to keys of its own sequence; with
 * Sq_i queries and Sk_i >= Sq_i keys, query r of the sequence sits at position
 * Sk_i - Sq_i + r and (causal) sees its keys j <= Sk_i - Sq_i + r (packed
 * self-attention: cu_seqlens_q = cu_seqlens_k).
 *   q, o [Hq,Tq,D], k, v [Hkv,Tk,D] (bf16, device), lse [Hq,Tq] (f32);
 *   cu_seqlens_q, cu_seqlens_k: DEVICE int32 [nseq + 1], nondecreasing, first 0,
 *   last Tq (resp. Tk); max_seqlen_q >= every Sq_i (sizes the grid).
 * K/V rows of other sequences never enter a result, but must be finite
 * (they meet a zero weight in the P V product).
 * Errors: GQA_ERR_INVALID_ARG on the host for null or misaligned pointers,
 * nseq, Tq, Tk < 1 or max_seqlen_q outside [1, Tq]; sizes as gqa_attn_fwd.
 * The bounds themselves live on the device and are checked there: a sequence
 * whose bounds are out of range, decreasing, have more queries than keys or
 * more than max_seqlen_q queries is skipped and gqa_attn_get_error() reports
 * GQA_ERR_INVALID_ARG.
 * Passage: RustingBrain docs, "Training infrastructure" (batches of token
 * windows); tang page, "An LLM" (prefill 512).
 */
int gqa_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, int nseq, int max_seqlen_q, int Hq, int Hkv, int Tq, int Tk, int D,
                        int causal, float scale, void* stream);

/*
 * Size in bytes of the device workspace gqa_attn_bwd needs (256-byte aligned
 * sections: the per-row D = rowsum(dO * O) and the scaled LSE, f32
 * [B,Hq,ceil(S/128)*128] each, and the f32 dQ accumulator [B,Hq,S,D]).
 * Returns 0 for arguments gqa_attn_bwd would reject.
 */
size_t gqa_attn_bwd_workspace_size(int B, int Hq, int Hkv, int S, int D);

/*
 * Backward of gqa_attn_fwd for the loss sum(O * dO).
 *   q, k, v, o, dO (bf16, device) and lse (f32, device) as produced/consumed by
 *   gqa_attn_fwd with the same causal and scale;
 *   dq [B,Hq,S,D], dk, dv [B,Hkv,S,D] (outputs, bf16, device). dk and dv are
 *   summed over the Hq/Hkv query heads that share each KV head; they are
 *   bitwise deterministic. dq is accumulated in f32 by reduce-add, so its
 *   last bits may differ between runs.
 *   workspace: device memory of at least gqa_attn_bwd_workspace_size() bytes,
 *   256-byte aligned, owned by the caller, not read before being written; it
 *   may be reused once the stream has passed this call.
 * Steps: D = rowsum(dO * O); recompute P from Q, K and LSE; dV = P^T dO;
 * dP = dO V^T; dS = P * (dP - D); dK = scale dS^T Q; dQ = scale dS K.
 * Passage: aiinsiders.net, "A compiler that derives GPU kernels matches
 * hand-tuned code" (the gradient through a comprehension is a comprehension;
 * the fused backward must meet the f32 tolerance).
 */
int gqa_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int S,
                 int D, int causal, float scale, void* stream);

/*
 * Decode: attention of Sq new query rows against a key/value cache of Sk >= Sq
 * rows (KV-cached decoding / prefill over a cache).
 *   q [B,Hq,Sq,D] (bf16, device): the new queries, query i at absolute
 *     position Sk - Sq + i; k_cache, v_cache [B,Hkv,Sk,D] (bf16, device);
 *   o [B,Hq,Sq,D] (bf16, device), lse [B,Hq,Sq] (f32, device) as in gqa_attn_fwd.
 *   causal: key j visible to query i iff j <= Sk - Sq + i (bottom-right).
 *   num_splits: number of key chunks processed in parallel (<= 0: chosen
 *     from the device's SM count); the chunk states are merged with the
 *     associative (m, l, acc) combine.
 *   workspace: device memory of gqa_attn_decode_workspace_size() bytes (same
 *     num_splits), 256-byte aligned, owned by the caller (per-chunk partials
 *     and one arrival counter per (batch, KV head), which the call zeroes
 *     itself; its contents need no initialisation). The CTA that finishes the
 *     last chunk of a (batch, KV head) merges the chunks in chunk order: one
 *     kernel (after a small memset), and the same result whichever CTA is last.
 * Supported: D in {64, 128}; (Hq/Hkv) * Sq <= 16 query rows per KV head.
 * Errors as gqa_attn_fwd; GQA_ERR_UNSUPPORTED for more than 16 rows per KV head.
 * Passage: RustingBrain docs, "Training infrastructure" (KV-cached decoding);
 * tang page, "How tang works" section 3 (the combine is associative, so the
 * key range splits and the parts recombine).
 */
size_t gqa_attn_decode_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, int num_splits);
int gqa_attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                        void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                        int causal, float scale, int num_splits, void* stream);

/*
 * Deterministic backward: the same arguments, workspace and results as
 * gqa_attn_bwd, but dQ is bitwise reproducible. A query-major kernel computes
 * each 128-row dQ tile in one CTA, in a fixed key order (recomputing S and dP
 * per (query, key) pair: 14 D flops per pair for the whole backward instead of
 * 10 D), and the KV-major kernel computes only dK and dV. No f32 dQ
 * accumulator is used (the workspace's dQ section is left untouched).
 * Passage: aiinsiders.net, "A compiler that derives GPU kernels matches
 * hand-tuned code" (the backward as a comprehension); the atomic-free dQ split
 * is the alternative to the f32 reduce-add named with the fused backward.
 */
int gqa_attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                               const float* lse, void* dq, void* dk, void* dv, void* workspace,
                               size_t workspace_bytes, int B, int Hq, int Hkv, int S, int D, int causal, float scale,
                               void* stream);

/*
 * Rotary position embedding fused with the attention (rotate-half pairing):
 * for position p and 0 <= i < D/2 the plane (x[i], x[i + D/2]) of every query
 * and key row turns by the angle with cosine rope_cos[p, i] and sine
 * rope_sin[p, i]; V is not rotated. The tables are f32 [S, D/2], device,
 * 16-byte aligned, owned by the caller (any base, scaling or offset).
 * gqa_attn_fwd_rope: O, LSE of attention over the rotated q and k (q, k, v, o,
 *   lse as gqa_attn_fwd). Queries are rotated as they land in shared memory;
 *   keys, which every query tile of their group re-reads, are rotated once
 *   into the workspace (>= gqa_attn_fwd_rope_workspace_size bytes, 256-byte
 *   aligned, caller-owned).
 * gqa_attn_bwd_rope: dq, dk (with respect to the UNROTATED q, k) and dv for the
 *   O, LSE of gqa_attn_fwd_rope. Queries are rotated once into the workspace
 *   (>= gqa_attn_bwd_rope_workspace_size bytes), keys as they land in shared
 *   memory; dK is turned back by the transposed rotation in the main kernel's
 *   epilogue and dQ in its f32-to-bf16 conversion.
 * Errors as gqa_attn_fwd / gqa_attn_bwd; GQA_ERR_INVALID_ARG for null or
 * misaligned tables; GQA_ERR_WORKSPACE_TOO_SMALL. Dense self-attention only.
 * Passage: tang page, "A transformer" (RMSNorm, RoPE, GQA attention, SwiGLU,
 * forward and backward); RustingBrain docs, "What is in the box" (rotary
 * positions).
 */
size_t gqa_attn_fwd_rope_workspace_size(int B, int Hkv, int S, int D);
int gqa_attn_fwd_rope(const void* q, const void* k, const void* v, const float* rope_cos, const float* rope_sin,
                      void* o, float* lse, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int S,
                      int D, int causal, float scale, void* stream);
size_t gqa_attn_bwd_rope_workspace_size(int B, int Hq, int Hkv, int S, int D);
int gqa_attn_bwd_rope(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      const float* rope_cos, const float* rope_sin, void* dq, void* dk, void* dv, void* workspace,
                      size_t workspace_bytes, int B, int Hq, int Hkv, int S, int D, int causal, float scale,
                      void* stream);

/*
 * Size in bytes of the device workspace gqa_attn_bwd_varlen needs for Hq query
 * heads over T packed rows (256-byte aligned sections: D and LSE*log2(e) rows,
 * f32 [Hq*T + 256] each, then the f32 dQ accumulator [Hq, T, D]).
 * Returns 0 for unsupported sizes.
 */
size_t gqa_attn_bwd_varlen_workspace_size(int Hq, int Hkv, int T, int D);

/*
 * Backward of packed self-attention over variable-length sequences: the
 * gradients of L = sum(O * dO) for the forward of gqa_attn_fwd_varlen with
 * cu_seqlens_q = cu_seqlens_k = cu_seqlens (each sequence attends only to
 * itself; causal: query r of a sequence sees its keys j <= r).
 *   q, o, dO, dq [Hq,T,D], k, v, dk, dv [Hkv,T,D] (bf16, device), lse [Hq,T]
 *   (f32, as the forward wrote it); cu_seqlens: DEVICE int32 [nseq + 1],
 *   nondecreasing, first 0, last T; max_seqlen >= every sequence's length.
 * dK, dV are summed over each KV head's query heads inside one CTA (bitwise
 * deterministic); dQ accumulates in f32 in the workspace (caller-owned,
 * 256-byte aligned, >= gqa_attn_bwd_varlen_workspace_size bytes).
 * Errors: as gqa_attn_bwd on the host (plus nseq, T < 1, max_seqlen outside
 * [1, T]); device-side bounds are checked as in gqa_attn_fwd_varlen (invalid
 * sequences skipped, GQA_ERR_INVALID_ARG from gqa_attn_get_error()).
 * Passage: aiinsiders.net, "A compiler that derives GPU kernels matches
 * hand-tuned code" (the backward as a comprehension, f32 accumulation);
 * RustingBrain docs, "Training infrastructure" (batches of token windows).
 */
int gqa_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                        void* dq, void* dk, void* dv, const int* cu_seqlens, int nseq, int max_seqlen, void* workspace,
                        size_t workspace_bytes, int Hq, int Hkv, int T, int D, int causal, float scale,
                        void* stream);

/*
 * Synchronises `stream`, then reads and clears the status word of `stream` on
 * the current device: the bits raised by kernels this library launched on
 * that stream since the last call. Work on other streams is neither waited
 * for nor reported (each of the first GQA_STATUS_STREAMS - 1 streams that call
 * into the library on a device has a word of its own; streams beyond that
 * share one word, and any of them may report, and clear, the others' bits).
 * Returns GQA_OK, GQA_ERR_TIMEOUT if a kernel gave up on a wait,
 * GQA_ERR_INTERNAL if a kernel's own shared-memory alignment check failed (it
 * then returned without work), GQA_ERR_INVALID_ARG if a packed batch's
 * device-side sequence bounds were invalid (those sequences were skipped),
 * GQA_ERR_BOUNDS (debug build only) if a coordinate check failed (the access
 * was skipped), or GQA_ERR_CUDA if the stream reports an error.
 */
int gqa_attn_get_error(void* stream);

/* Static, human-readable text of an error code. Never NULL. */
const char* gqa_attn_strerror(int code);

/* The CUDA error code behind the last GQA_ERR_CUDA returned on this host thread (0 if none). */
int gqa_attn_last_cuda_error(void);

/*
 * Backward without caller-provided workspace and without any allocation (the
 * paper has no counterpart; this is a convenience of this library).
 *
 * For callers that cannot call cudaMalloc: code running where device
 * allocation is forbidden or unsafe (inside an allocator's own callbacks, in
 * a framework that owns all device memory and hands out only tensors, on
 * hosts that must not allocate after start-up). The backward's scratch
 * memory (D and scaled-LSE rows, f32 dQ accumulator) lives instead in one
 * file-scope device array of GQA_NOALLOC_SCRATCH_BYTES (64 MiB) that every
 * device which loads the library holds until the process exits.
 * Arguments, layout, outputs and errors are those of gqa_attn_bwd without the
 * workspace pair. Problems whose workspace (gqa_attn_bwd_workspace_size)
 * exceeds the array are rejected with GQA_ERR_WORKSPACE_TOO_SMALL; invalid
 * sizes with GQA_ERR_INVALID_ARG / GQA_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.
 * Every call on a device shares the array and it keeps the last call's
 * contents; each call rewrites everything it reads (the dQ accumulator is
 * zeroed by the call itself). Calls that overlap on the GPU (concurrent
 * streams or host threads on the same device) race on the array.
 * Calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (64u << 20)
int gqa_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int D,
                         int causal, float scale, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
