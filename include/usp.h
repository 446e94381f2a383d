/*
 * usp.h -- C ABI of libusp: the attention step of a diffusion transformer
 * under USP (Ulysses x Ring) sequence parallelism, with the rank grid of
 * ulysses x ring virtual ranks simulated on ONE GPU (GB300, sm_103a).
 *
 * Sources (web pages, by title):
 *  [HB] "Multi-GPU parallelism: spreading one step over several cards",
 *       section "Sequence parallelism: Ulysses and Ring": the Ulysses
 *       all-to-all (per-card token slices <-> per-card head groups), per-card
 *       attention, and the Ring step that combines per-KV-block results by a
 *       log-sum-exp merge (the online-softmax rule).
 *  [PR] "Feat: USP sequence parallelism (Ulysses x Ring) via
 *       SequenceParallelPlan; Wan enabled": Design ("Coordinates": sp =
 *       ulysses x ring, Ulysses ranks contiguous, ring ranks strided; "Ring
 *       kernel selection": the ring kernels also produce the log-sum-exp and have
 *       matching backward kernels),
 *       Limitations (the conditions that must fail loudly), Numerics.
 *  [VO] vllm-omni "Parallelism Acceleration Guide": sequence chunked by SP
 *       rank in rank order; hybrid sp = ulysses_degree x ring_degree.
 *
 * Conventions shared by every call
 * --------------------------------
 *  * All tensor pointers are DEVICE pointers on the current CUDA device,
 *    owned by the caller; the library never allocates, frees or retains
 *    them.  Buffers that a call writes must not overlap buffers it reads.
 *  * Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and returns after enqueueing its kernels.
 *  * Arguments are validated on the host BEFORE anything is enqueued; an
 *    invalid call enqueues nothing and returns a USP_ERR_* code.  An empty
 *    problem (a zero B, H or row count where allowed) enqueues nothing and
 *    returns USP_OK.
 *  * Pointers handed to the tensor-core (bf16) paths must be 16-byte
 *    aligned (tensor-memory-accelerator copies); misaligned pointers return
 *    USP_ERR_INVALID_ARG.
 *  * Device-side waits are bounded.  If one expires the kernel records it in
 *    a per-device error word and returns early (outputs are then undefined);
 *    usp_device_status() reports it.  No kernel traps or asserts.
 *  * Layouts (row-major, innermost last):
 *      plain           [B, H, N, D]
 *      token-sharded   [ring, ulysses, B, H, Ns, D], Ns = N/(ulysses*ring):
 *                      virtual rank (g, j) -- ring index g, Ulysses index j,
 *                      sp_rank = g*ulysses + j -- holds tokens
 *                      [sp_rank*Ns, (sp_rank+1)*Ns) of every head ([PR]
 *                      Coordinates; [VO] chunk by rank).  With
 *                      ulysses = ring = 1 this is the plain layout.
 *      head-sharded    [ring, ulysses, B, H/ulysses, Nr, D], Nr = N/ring:
 *                      rank (g, j) holds heads [j*Hu, (j+1)*Hu) of the
 *                      tokens of ring group g, source ranks concatenated in
 *                      rank order ([HB] all_to_all_heads).
 *      LSE             one fp32 per (row, head): the layouts above without
 *                      the trailing D; natural logarithm.
 */
#ifndef USP_H
#define USP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* usp_stream_t; /* a cudaStream_t */

typedef enum { USP_F32 = 0, USP_BF16 = 1 } usp_dtype;

typedef enum {
  USP_MATERIALISED = 0, /* re-layout, per-(rank, ring step) attention, merge, re-layout back */
  USP_FUSED = 1         /* one kernel reading and writing the token-sharded stacks in place */
} usp_mode;

enum {
  USP_OK = 0,
  USP_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer, scale not finite */
  USP_ERR_DIVISIBILITY = 2, /* H % ulysses != 0 or N % (ulysses*ring) != 0 ([PR] Limitations) */
  USP_ERR_UNSUPPORTED = 3,  /* dtype / head dim combination without a kernel */
  USP_ERR_WORKSPACE = 4,    /* workspace null or smaller than usp_attention_workspace_bytes() */
  USP_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed; see usp_last_cuda_error() */
  USP_ERR_TIMEOUT = 6       /* a bounded device-side wait expired (usp_device_status) */
};

/* Ulysses all-to-all, token -> head, as an on-device re-layout ([HB]
 * all_to_all_heads; [PR] Design, usp_attention's first step).
 *   dst[g, j, b, h', s*Ns + n, d] = src[g, s, b, j*Hu + h', n, d]
 * src: token-sharded stack [ring, ulysses, B, H, Ns, D]; dst: head-sharded
 * stack [ring, ulysses, B, Hu, Nr, D].  Pure indexing, bit-exact, any
 * element type of `dtype`'s width; for the LSE pass USP_F32 with D = 1.
 * Errors: INVALID_ARG (null, negative size, ulysses/ring < 1),
 * DIVISIBILITY (H % ulysses, N % (ulysses*ring)), CUDA. */
int usp_relayout_tok2head(const void* src, void* dst, int64_t B, int64_t H, int64_t N, int64_t D,
                          int ulysses, int ring, usp_dtype dtype, usp_stream_t stream);

/* The inverse re-layout, head -> token ([HB] all_to_all_tokens).
 *   dst[g, s, b, j*Hu + h', n, d] = src[g, j, b, h', s*Ns + n, d]
 * Same arguments, errors and layouts with src and dst exchanged. */
int usp_relayout_head2tok(const void* src, void* dst, int64_t B, int64_t H, int64_t N, int64_t D,
                          int ulysses, int ring, usp_dtype dtype, usp_stream_t stream);

/* Attention of one (query block, KV chunk) pair, returning the output and
 * the log-sum-exp ([HB] per-card attention; [PR] "Ring kernel selection":
 * kernels return LSE).  For every (b, h) and query row i:
 *   S_ij = scale * q_i . k_j,  lse_i = ln sum_j exp(S_ij),
 *   out_i = sum_j exp(S_ij - lse_i) v_j.
 * No mask, not causal, no dropout.  q, out: [B, H, Nq, D]; k, v:
 * [B, H, Nk, D], all in `dtype`; lse: [B, H, Nq] fp32.  bf16 runs on the
 * tcgen05 tensor cores with fp32 accumulation (D = 128); fp32 runs on the
 * FP32 pipes in full fp32 (D <= 128).
 * Errors: INVALID_ARG (null, Nk < 1, negative size, non-finite scale,
 * misaligned), UNSUPPORTED (head dim), CUDA. */
int usp_attn_chunk_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                       int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale,
                       usp_dtype dtype, usp_stream_t stream);

/* The Ring step's log-sum-exp merge of R partial results over disjoint KV
 * chunks ([HB] Ring paragraph; the formula is the standard one):
 *   m = max_t lse_t,  lse = m + ln sum_t exp(lse_t - m),
 *   out = sum_t exp(lse_t - lse) * out_t
 * outs: R contiguous [B, H, Nq, D] blocks in `dtype`; lses: R contiguous
 * [B, H, Nq] fp32 blocks; out: [B, H, Nq, D] `dtype`; lse: [B, H, Nq] fp32.
 * Arithmetic in fp32.  Errors: INVALID_ARG (null, R < 1), CUDA. */
int usp_lse_merge(const void* outs, const float* lses, int R, void* out, float* lse,
                  int64_t B, int64_t H, int64_t Nq, int64_t D, usp_dtype dtype, usp_stream_t stream);

/* Bytes of workspace usp_attention_fwd (backward = 0) or the backward
 * (backward = 1: usp_attention_bwd with USP_FUSED, usp_attention_bwd_materialised
 * with USP_MATERIALISED, which also covers usp_attention_bwd) needs for this
 * problem; 0 when none is needed.  Returns 0 as well for arguments the call
 * itself would reject. */
size_t usp_attention_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D, int ulysses, int ring,
                                     usp_dtype dtype, usp_mode mode, int backward);

/* USP attention forward over `ulysses` x `ring` virtual ranks ([PR] Design:
 * Ulysses all-to-all, then the Ring steps with an LSE-returning kernel, then
 * the all-to-all back).  q, k, v, out: token-sharded stacks
 * [ring, ulysses, B, H, Ns, D]; lse: [ring, ulysses, B, H, Ns] fp32.
 * The result equals unsharded attention of the re-assembled sequence.
 *   USP_MATERIALISED: tok2head(q,k,v) -> for every rank (g, j) and ring step
 *     t the chunk attention against KV chunk (g - t) mod ring -> merge over
 *     t -> head2tok(out, lse).  Partial outputs are stored in `dtype`.  With
 *     ring > 1 the merge writes each merged row straight to its token-sharded
 *     place (merge and head2tok in one pass); with ring = 1 the chunk result
 *     is re-laid out head -> token.
 *     Needs usp_attention_workspace_bytes() of workspace.
 *   USP_FUSED: one kernel reads q, k, v in place and keeps the ring merge
 *     in registers (online softmax over every KV chunk); no workspace.
 * Errors: INVALID_ARG, DIVISIBILITY, UNSUPPORTED, WORKSPACE, CUDA. */
int usp_attention_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      int64_t B, int64_t H, int64_t N, int64_t D, int ulysses, int ring, float scale,
                      usp_dtype dtype, usp_mode mode, void* workspace, size_t workspace_bytes,
                      usp_stream_t stream);

/* USP attention backward ([PR] Numerics: the Ulysses exchange only moves
 * data, so the gradients take the inverse exchange; each ring step uses its
 * own KV chunk and the MERGED lse).  With P = exp(scale q k^T - lse):
 *   dV = P^T dO, dP = dO V^T, Delta_i = sum_d dO_id O_id,
 *   dS = P * (dP - Delta), dQ = scale dS K, dK = scale dS^T Q.
 * q, k, v, out, dout, dq, dk, dv: token-sharded stacks in `dtype`; lse: the
 * forward's fp32 LSE.  Needs usp_attention_workspace_bytes(..., 1).
 * The bf16 path runs its dQ kernel concurrently with the dK/dV kernel on a
 * library-owned stream of the current device, forked from and joined back to
 * `stream` with events (so the call stays ordered on `stream` and can be
 * captured into a CUDA graph); concurrent calls on one device take turns on
 * that stream.
 * Errors: as usp_attention_fwd. */
int usp_attention_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t N,
                      int64_t D, int ulysses, int ring, float scale, usp_dtype dtype, void* workspace,
                      size_t workspace_bytes, usp_stream_t stream);

/* The same backward through the materialised Ulysses path ([PR] Numerics:
 * the Ulysses exchange only moves data, so the gradients take the inverse
 * exchange; each ring step uses its own KV chunk and the merged lse):
 *   tok2head(q, k, v, O, dO) in one launch and tok2head(lse) ->
 *   per (ring rank g, Ulysses rank j, ring step t) the chunk backward of
 *   query chunk g against KV chunk (g - t) mod ring over the head-sharded
 *   stacks, dQ summed over t and dK/dV summed over the query chunks ->
 *   head2tok(dq, dk, dv) in one launch.
 * Same arguments, layouts and results as usp_attention_bwd (the sums run
 * in another order, so results agree to rounding, not bit for bit).
 * Needs usp_attention_workspace_bytes(..., USP_MATERIALISED, 1): eight
 * head-sharded tensors plus the lse and two per-row vectors.  The bf16 path
 * forks its dQ kernel as usp_attention_bwd does.
 * Errors: as usp_attention_bwd. */
int usp_attention_bwd_materialised(const void* q, const void* k, const void* v, const void* out,
                                   const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                   int64_t B, int64_t H, int64_t N, int64_t D, int ulysses, int ring,
                                   float scale, usp_dtype dtype, void* workspace, size_t workspace_bytes,
                                   usp_stream_t stream);

/* Bytes of workspace usp_attention_fwd_joint needs (0 for USP_FUSED);
 * with_text_queries = 1 when q_txt will be given.  Returns 0 as well for
 * arguments the call itself would reject. */
size_t usp_attention_joint_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t Nt, int64_t D, int ulysses,
                                           int ring, usp_dtype dtype, usp_mode mode, int with_text_queries);

/* Joint text + image USP attention forward ([VO] "How to parallelize a new
 * model": a dual-stream model attends over the concatenated text and image
 * sequences; image tokens are chunked across the SP ranks, text embeddings
 * stay replicated on every rank).  Image tensors q, k, v, out, lse are the
 * token-sharded stacks of usp_attention_fwd; text tensors k_txt, v_txt (and
 * q_txt, out_txt) are plain [B, H, Nt, D] in `dtype`, lse_txt [B, H, Nt] fp32,
 * the same on every virtual rank.  The result equals unsharded attention of
 * every query over the Nt text + N image keys of its head.
 *   USP_MATERIALISED: tok2head(q,k,v) -> per rank (g, j) the ring chunk
 *     partials (as usp_attention_fwd) plus one partial against the text K/V
 *     of head group j -> merge of ring + 1 partials written straight to the
 *     token-sharded out, lse (the merge and head2tok in one pass).  Text
 *     queries of head group j: one partial per ring chunk c of that group
 *     (the same on every ring rank, computed once) plus one against the
 *     text K/V -> merge into out_txt, lse_txt.  The launch of the partials
 *     against the text runs on the library-owned stream of the current
 *     device that usp_attention_bwd uses, forked from and joined back to
 *     `stream` with events (the call stays ordered on `stream`).
 *   USP_FUSED: one kernel launch reads the stacks and the text in place
 *     (image and text queries share it); the text K/V are the last KV tiles
 *     of the online softmax.
 * q_txt may be NULL (no text queries: out_txt, lse_txt are then ignored).
 * Nt = 0 is usp_attention_fwd.
 * Errors: INVALID_ARG (null, negative Nt, misaligned, non-finite scale),
 * DIVISIBILITY, UNSUPPORTED, WORKSPACE, CUDA. */
int usp_attention_fwd_joint(const void* q, const void* k, const void* v, const void* q_txt, const void* k_txt,
                            const void* v_txt, void* out, float* lse, void* out_txt, float* lse_txt, int64_t B,
                            int64_t H, int64_t N, int64_t Nt, int64_t D, int ulysses, int ring, float scale,
                            usp_dtype dtype, usp_mode mode, void* workspace, size_t workspace_bytes,
                            usp_stream_t stream);

/* Cross-attention under sequence parallelism ([PR]: replicated K/V make
 * local attention exact and it follows the stock path; [VO] "How to
 * parallelize a new model": text embeddings stay replicated on every SP
 * rank).  q, out: token-sharded image stacks [ring, ulysses, B, H, Ns, D];
 * lse: [ring, ulysses, B, H, Ns] fp32; k_txt, v_txt: plain [B, H, Nt, D],
 * the same on every virtual rank.  Every rank attends its own query tokens to
 * the complete text K/V: one kernel launch, no re-layout, no merge.  The
 * result equals unsharded attention of the image queries against the text.
 * Errors: INVALID_ARG (null, Nt < 1, misaligned, non-finite scale),
 * DIVISIBILITY (N % (ulysses*ring)), UNSUPPORTED, CUDA. */
int usp_cross_attention_fwd(const void* q, const void* k_txt, const void* v_txt, void* out, float* lse,
                            int64_t B, int64_t H, int64_t N, int64_t Nt, int64_t D, int ulysses, int ring,
                            float scale, usp_dtype dtype, usp_stream_t stream);

/* FP8 (OCP E4M3) per-head quantisation ([HB] Wan latency table: "FP8 low
 * precision" as the last latency step; the pages print no scheme, this is
 * the plainest one).  x: bf16 token-sharded stack [ring, ulysses, B, H, Ns,
 * D]; x8: uint8 codes in the same layout; scales: [B, H] fp32.  Per (b, h)
 * head over every shard, token and dimension: amax = max |x|,
 * code = e4m3(x * (448 / amax)) (fp32 multiply and divide, round to nearest
 * even, saturating at +-448), scales = amax / 448; an all-zero head gets
 * scale 1 and zero codes.  x must be finite.  D % 16 == 0; 16-byte aligned
 * pointers.  Errors: INVALID_ARG, DIVISIBILITY, UNSUPPORTED, CUDA. */
int usp_quantize_e4m3(const void* x, void* x8, float* scales, int64_t B, int64_t H, int64_t N, int64_t D,
                      int ulysses, int ring, usp_stream_t stream);

/* Bytes of workspace usp_attention_fwd_fp8 needs (0 for arguments it would
 * reject): the E4M3 codes of q and k, the transposed codes of v (keys padded
 * to a multiple of 16 per shard) and the per-head amax of all three. */
size_t usp_attention_fp8_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D, int ulysses, int ring);

/* FP8 fused USP attention forward.  q, k, v, out: bf16 token-sharded stacks
 * as in usp_attention_fwd (D = 128); lse: fp32.  q, k and v are quantised
 * per head as in usp_quantize_e4m3; Q K^T and P V run on the tensor cores
 * in E4M3 with fp32 accumulation (P rounded to E4M3 for the product, its row
 * sum kept in fp32); the softmax is fp32; the output is dequantised to bf16.
 * The result approximates usp_attention_fwd; against attention of the
 * dequantised q, k, v the remaining error is that of rounding P (bounded
 * statistically, not element-wise).
 * Errors: INVALID_ARG, DIVISIBILITY, UNSUPPORTED (D != 128), WORKSPACE, CUDA. */
int usp_attention_fwd_fp8(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B, int64_t H,
                          int64_t N, int64_t D, int ulysses, int ring, float scale, void* workspace,
                          size_t workspace_bytes, usp_stream_t stream);

/* The materialised forward (same arguments, layouts, result and errors as
 * usp_attention_fwd with mode USP_MATERIALISED) for callers that cannot
 * allocate device memory: code running under a framework whose caching
 * allocator owns the card, where an extra cudaMalloc can fail or break the
 * memory budget, and latency-critical callers that must not call
 * cudaMalloc/cudaFree (which may synchronise the device) on their request
 * path.  The pages have no counterpart to this call; it exists for such hosts.
 * Its scratch is one 64 MiB array compiled into the library (every device that
 * loads libusp holds it until exit).  Arguments are checked as
 * usp_attention_fwd checks them, in the same order; a valid problem whose
 * workspace (usp_attention_workspace_bytes) exceeds 64 MiB then returns
 * USP_ERR_WORKSPACE.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current and caches it with
 * the context's id; make that first call before any stream capture.  After a
 * cudaDeviceReset the next call on that device looks the address up again
 * (so that call, too, belongs outside a capture).  All calls share the array and it keeps the last call's
 * contents (nothing here needs it zeroed); calls that overlap on the GPU --
 * other streams or host threads -- race on it and must be serialised by the
 * caller.  Allocates nothing. */
int usp_attention_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B,
                              int64_t H, int64_t N, int64_t D, int ulysses, int ring, float scale,
                              usp_dtype dtype, usp_stream_t stream);

/* Phase timing for profiling: while enabled (enable = 1), each later
 * usp_attention_fwd / usp_attention_bwd call on this thread records a CUDA
 * event on its stream before its first kernel and after each kernel group:
 *   fused forward:        [attention]
 *   materialised forward: [tok2head q,k,v] [chunk attention]
 *                         [ring > 1: merge into the token-sharded out and lse |
 *                          ring = 1: head2tok of out and lse (one launch when
 *                          Ns % 4 == 0)]
 *   bf16 backward:        [Delta/lse prep] [dK,dV kernel] [dQ kernel]
 *                         (the two kernels run concurrently; both phases
 *                         are timed from the end of the prep)
 *   bf16 materialised backward: [tok2head q,k,v,O,dO and lse] [prep]
 *                         [dK,dV kernel] [dQ kernel] [join: end of dQ to
 *                         the end of both] [head2tok dq,dk,dv]
 *   FP8 forward:          [quantise q, k, v] [FP8 attention]
 *   joint fused:          [attention: image and text queries, one launch]
 *   joint materialised:   [tok2head q,k,v] [partials against the image chunks
 *                         and against the text] [merge into the token-sharded
 *                         out and lse] [text-query merge]
 * (the fp32 fused forward and usp_attention_bwd record nothing; the fp32
 * materialised backward records [tok2head] [backward] [head2tok]).  The events
 * are created by the library on first enable; enabling starts a fresh
 * record, disabling keeps the most recent call's record readable.  While
 * enabled, the events between a call's kernels also stop each kernel from
 * starting under the previous one's tail.  Returns USP_OK or USP_ERR_CUDA. */
int usp_profile_phases(int enable);

/* Waits for the last event of the most recent recorded call on this thread
 * and writes the milliseconds of each of its phases to ms[0 .. n-1]; returns
 * n (<= max_phases), 0 if nothing was recorded, or -USP_ERR_CUDA. */
int usp_profile_read(float* ms, int max_phases);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns USP_OK, USP_ERR_TIMEOUT if a bounded device wait expired
 * since the last call, or USP_ERR_CUDA. */
int usp_device_status(usp_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* usp_status_string(int status);

/* The cudaError_t of the last USP_ERR_CUDA return on this thread (0 if none). */
int usp_last_cuda_error(void);

/* Test hook: the number of polls a device-side wait may make before it
 * gives up (negative restores the default).  0 makes every wait that is not
 * already satisfied expire, so the timeout path runs without any hang.
 * Applies to launches enqueued after the call, on every device. */
void usp_set_debug_spin_limit(long long polls);

/* The same hook under its earlier name (kept for existing callers). */
void usp_set_spin_limit(long long polls);

#ifdef __cplusplus
}
#endif

#endif /* USP_H */
