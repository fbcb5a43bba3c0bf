/*
 * msa.h -- C ABI of libmsa.so: MiniMax-M3 MSA block-sparse attention on one
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes is defined on these pages:
 *   "MiniMax-M3.1-Flash" (miles docs), section 1 "Model Introduction":
 *       a 4-head indexer (dim 128, its own gemma q/k norm and RoPE) scores every
 *       causal 128-token key block by its maximum logit; each query attends to
 *       the 16 best blocks, its own block always included; index head h picks
 *       the blocks of KV head h.  Attention is GQA, 64 query / 4 KV heads of
 *       dim 128, with per-head gemma q/k norm and RoPE on the first 64 dims
 *       (base 1e7).
 *   same page, section 5.1 "Parallelism": the sparse attention runs on
 *       THD-packed sequences (cu_seqlens).
 *   same page, section 5.4 "Notable quirks": the indexer is frozen, so the
 *       block selection gets no gradient.
 *   "[1/4] Add MiniMax-M3 support - #4581" (radixark/miles), "Kernel tuning":
 *       per-block max-logit scores, top-k select, forward and dQ/dK/dV
 *       backward of the block-sparse attention kernel.
 *   "MiniMax-M3" (Megatron-Bridge docs), "Architecture Notes": Gemma-style
 *       RMSNorm x * (1 + w); "Known Limitations": 16 x 128 = 2048 keys per
 *       query, so the method equals full causal attention up to that length.
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer (cudaMalloc / torch CUDA
 *     tensor memory), 16-byte aligned, contiguous in the stated layout, on
 *     the device that is current when the call is made.
 *   - bf16 means IEEE bfloat16 (2 bytes); compute is fp32 inside the kernels.
 *   - D (head dim) is 128, the key block is 128 tokens, top-k is 16, the
 *     rotated part is the first 64 channels: the library rejects other values.
 *   - Packed (THD) inputs: token t of the pack belongs to sequence s with
 *     cu_seqlens[s] <= t < cu_seqlens[s+1]; its position is t - cu_seqlens[s].
 *     Key block b of sequence s covers positions [128 b, 128 b + 128); the last
 *     block of a sequence may be partial.  cu_seqlens is int32 [S + 1] on the
 *     device, cu_seqlens[0] = 0, non-decreasing, cu_seqlens[S] = T, and no
 *     sequence longer than max_seqlen.  The library does not read device
 *     memory on the host, so it cannot verify these contents: kernels clamp
 *     indices and set MSA_STATUS_BOUNDS in the device status word instead of
 *     reading or writing out of range.
 *   - Selected block ids (sel) are int32 [T, H, 16], relative to the start of
 *     the token's sequence, sorted ascending, padded with -1.
 *   - GQA: query head i uses KV head i / (Hq / Hkv).
 *   - Ownership: the caller allocates every buffer, including the workspace
 *     (size from the matching *_workspace_size call, 256-byte aligned).  The
 *     library never allocates or frees device memory and never synchronizes
 *     the stream.  Outputs are fully overwritten.  Two calls that may run at
 *     the same time need distinct workspaces.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Errors: argument checks run on the host before any launch and return
 *     MSA_ERR_INVALID_ARG / MSA_ERR_UNSUPPORTED with nothing enqueued; a
 *     failed launch returns MSA_ERR_CUDA.  msa_last_error() gives the message
 *     of the calling thread's last failure.  Kernels never trap: a wait that
 *     runs out or an index out of range sets a bit in the device status word,
 *     read (and cleared) by msa_check_status().
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MSA_API __attribute__((visibility("default")))
#else
#define MSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or workspace */
  MSA_ERR_UNSUPPORTED = 2,  /* a shape the library does not implement */
  MSA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  MSA_ERR_TIMEOUT = 4,      /* msa_check_status: a kernel wait ran out */
  MSA_ERR_BOUNDS = 5        /* msa_check_status: an index was out of range */
} msa_status_t;

/* A cudaStream_t passed through as an opaque handle. */
typedef void* msa_stream_t;

#define MSA_ABI_VERSION 1

MSA_API int msa_abi_version(void);

/* Message of the calling thread's most recent failed call ("" if none). */
MSA_API const char* msa_last_error(void);

/* Synchronizes `stream`, then reads and clears the device status word of the
 * current device.  MSA_OK if no kernel reported a problem since the last
 * check, MSA_ERR_TIMEOUT or MSA_ERR_BOUNDS otherwise.  Meant for tests and
 * debugging; it blocks the host. */
MSA_API msa_status_t msa_check_status(msa_stream_t stream);

/* Diagnostic of the failure-detection path: launches one kernel on `stream`
 * whose bounded wait on an mbarrier that nothing completes runs out (after the
 * library's wait limit, about 2 s) and sets the timeout bit of the status word,
 * then returns.  No fault is raised and the context stays usable; the next
 * msa_check_status returns MSA_ERR_TIMEOUT (wait site 65535). */
MSA_API msa_status_t msa_selftest_wait(msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Prologue ("MiniMax-M3.1-Flash", 1 "Model Introduction"; "MiniMax-M3",
 * "Architecture Notes").  x bf16 [T, H, 128] -> y bf16 [T, H, 128] (y may be
 * x itself, for an in-place update):
 *   y = x / sqrt(mean(x^2) + eps) * (1 + w)        per (token, head), w bf16 [128]
 *   then channels i and i + rope_dim/2 (i < rope_dim/2) are rotated by the
 *   angle pos * rope_base^(-2 i / rope_dim), pos = the token's in-sequence
 *   position; channels >= rope_dim pass through.  rope_dim must be 64.
 * The four-tensor form runs q [T,Hq,128], k [T,Hkv,128], q_idx and k_idx
 * [T,Hi,128] with their own weights in one launch; same result as four calls.
 * Head counts: 1 <= H <= 256 per tensor (MSA_ERR_INVALID_ARG below,
 * MSA_ERR_UNSUPPORTED above; nothing is enqueued).
 */
MSA_API msa_status_t msa_qk_norm_rope(const void* x, void* y, int T, int H, const void* w,
                                      const int32_t* cu_seqlens, int S, int rope_dim,
                                      float rope_base, float eps, msa_stream_t stream);

MSA_API msa_status_t msa_qk_norm_rope4(const void* q, void* q_out, int Hq, const void* k,
                                       void* k_out, int Hkv, const void* q_idx,
                                       void* q_idx_out, const void* k_idx, void* k_idx_out,
                                       int Hi, const void* w_q, const void* w_k,
                                       const void* w_qi, const void* w_ki,
                                       const int32_t* cu_seqlens, int S, int T, int rope_dim,
                                       float rope_base, float eps, msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Prologue backward (the gradients of msa_qk_norm_rope for one tensor; the
 * indexer's prologue needs none: "MiniMax-M3.1-Flash", 5.4 "Notable quirks").
 * x: the prologue's input, bf16 [T, H, 128]; dy = dL/dy for its output (same
 * shape, e.g. dq or dk from msa_sparse_attn_bwd).  With z = gemma_norm(x, w)
 * and y = RoPE(z):  dz = R^T dy (the rotation turned back), r =
 * 1/sqrt(mean(x^2) + eps), xh = x r, g = dz (1 + w):
 *   dx = r (g - xh mean(g xh))          bf16 [T, H, 128]  (dx may be dy)
 *   dw = sum over tokens and heads of dz * xh     fp32 [128] (overwritten)
 * dw is summed in a fixed order (run to run identical).  Workspace from
 * msa_qk_norm_rope_bwd_workspace_size; other arguments (and the head-count
 * limit 1 <= H <= 256) as for msa_qk_norm_rope.
 */
MSA_API size_t msa_qk_norm_rope_bwd_workspace_size(int T, int H);

MSA_API msa_status_t msa_qk_norm_rope_bwd(const void* x, const void* dy, void* dx, float* dw,
                                          int T, int H, const void* w,
                                          const int32_t* cu_seqlens, int S, int rope_dim,
                                          float rope_base, float eps, void* workspace,
                                          size_t workspace_bytes, msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Index select ("MiniMax-M3.1-Flash", 1 "Model Introduction"; "#4581",
 * "Kernel tuning").  q_idx, k_idx: post-prologue bf16 [T, Hi, 128].
 * For token t at position p and index head h the own block is p / 128; every
 * earlier block b of the sequence is scored by max_j q_idx[t,h] . k_idx[j,h]
 * over its keys (fp32 accumulation); the own block plus the best
 * min(15, own) earlier blocks (equal scores: lower id) are written to
 * sel [T, Hi, 16] (ascending, -1 padded).  topk must be 16.
 */
MSA_API size_t msa_index_select_workspace_size(int T, int S, int Hi, int max_seqlen);

MSA_API msa_status_t msa_index_select(const void* q_idx, const void* k_idx,
                              const int32_t* cu_seqlens, int S, int T, int Hi,
                              int max_seqlen, int topk, int32_t* sel, void* workspace,
                              size_t workspace_bytes, msa_stream_t stream);

/* The same selection with the "init" rule that "#4581" (Kernel tuning) names
 * beside the local and causal rules but does not define.  Read here as: the
 * first n_init blocks of every sequence (those before the token's own block)
 * are always kept; the best of the other earlier blocks fill the remaining
 * 15 - min(n_init, own) slots.  0 <= n_init <= 15; n_init = 0 is
 * msa_index_select.  Workspace: msa_index_select_workspace_size.
 */
MSA_API msa_status_t msa_index_select_ex(const void* q_idx, const void* k_idx,
                                 const int32_t* cu_seqlens, int S, int T, int Hi,
                                 int max_seqlen, int topk, int n_init, int32_t* sel,
                                 void* workspace, size_t workspace_bytes,
                                 msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Block-sparse attention forward ("MiniMax-M3.1-Flash", 1; "#4581").
 * q bf16 [T, Hq, 128]; k, v bf16 [T, Hkv, 128]; sel int32 [T, Hkv, 16].
 * For query head i of token t (KV head g = i / (Hq/Hkv)) the keys are those
 * of the blocks in sel[t, g] at positions <= the query's position:
 *   o[t, i]   = softmax(scale * q k_j) v_j            bf16 [T, Hq, 128]
 *   lse[t, i] = log sum_j exp(scale * q k_j)         fp32 [T, Hq] (natural log)
 * Hq / Hkv must divide 128.
 */
MSA_API size_t msa_sparse_attn_fwd_workspace_size(int T, int S, int Hq, int Hkv, int max_seqlen);

MSA_API msa_status_t msa_sparse_attn_fwd(const void* q, const void* k, const void* v,
                                 const int32_t* sel, const int32_t* cu_seqlens, int S,
                                 int T, int Hq, int Hkv, int max_seqlen, float scale,
                                 void* o, float* lse, void* workspace,
                                 size_t workspace_bytes, msa_stream_t stream);

/* The forward of a training step: msa_sparse_attn_fwd that also zeroes the
 * fp32 accumulators and item counters of `bwd_workspace` (sized by
 * msa_sparse_attn_bwd_workspace_size for the same T, S, Hq, Hkv, max_seqlen)
 * while it runs, by bulk copies from the forward's otherwise idle memory
 * bandwidth.  It stands in for msa_sparse_attn_bwd_prepare: follow it with
 * msa_sparse_attn_bwd_prepared on that workspace (same stream, or an event),
 * writing nothing into the workspace in between. */
MSA_API msa_status_t msa_sparse_attn_fwd_train(const void* q, const void* k, const void* v,
                                               const int32_t* sel, const int32_t* cu_seqlens,
                                               int S, int T, int Hq, int Hkv, int max_seqlen,
                                               float scale, void* o, float* lse,
                                               void* workspace, size_t workspace_bytes,
                                               void* bwd_workspace, size_t bwd_workspace_bytes,
                                               msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Block-sparse attention backward ("#4581", "Kernel tuning"; the selection
 * is constant: "MiniMax-M3.1-Flash", 5.4 "Notable quirks").
 * Inputs as for the forward plus o (bf16, the forward's output), dout (bf16
 * [T, Hq, 128], gradient of the loss w.r.t. o) and lse (fp32 [T, Hq]).
 * With P = exp(scale q k^T - lse) over the attended keys, dP = dout v^T and
 * Delta = rowsum(dout * o):  dS = P * (dP - Delta);
 *   dq = scale dS k  (bf16 [T,Hq,128]),  dk = scale dS^T q,  dv = P^T dout
 *   (bf16 [T,Hkv,128]; sums over all query heads and tokens using the key).
 */
MSA_API size_t msa_sparse_attn_bwd_workspace_size(int T, int S, int Hq, int Hkv, int max_seqlen);

MSA_API msa_status_t msa_sparse_attn_bwd(const void* q, const void* k, const void* v,
                                 const void* o, const void* dout, const float* lse,
                                 const int32_t* sel, const int32_t* cu_seqlens, int S,
                                 int T, int Hq, int Hkv, int max_seqlen, float scale,
                                 void* dq, void* dk, void* dv, void* workspace,
                                 size_t workspace_bytes, msa_stream_t stream);

/* The backward in two parts, so that a caller can clear the workspace's fp32
 * accumulators (about T * (Hq + 2 Hkv) * 512 bytes, one memset) while other
 * work runs, e.g. on a second stream during the forward:
 *   msa_sparse_attn_bwd_prepare  clears them on `stream` (same sizes as the
 *                                backward that follows);
 *   msa_sparse_attn_bwd_prepared is msa_sparse_attn_bwd without the clear.
 * The caller orders the prepare before the prepared call (same stream, or an
 * event) and writes nothing into the workspace in between; the prepared call
 * leaves the accumulators dirty, so every call needs its own prepare.
 * msa_sparse_attn_bwd equals prepare + prepared on one stream.
 */
MSA_API msa_status_t msa_sparse_attn_bwd_prepare(int T, int S, int Hq, int Hkv, int max_seqlen,
                                                 void* workspace, size_t workspace_bytes,
                                                 msa_stream_t stream);

MSA_API msa_status_t msa_sparse_attn_bwd_prepared(const void* q, const void* k, const void* v,
                                                  const void* o, const void* dout,
                                                  const float* lse, const int32_t* sel,
                                                  const int32_t* cu_seqlens, int S, int T,
                                                  int Hq, int Hkv, int max_seqlen, float scale,
                                                  void* dq, void* dk, void* dv, void* workspace,
                                                  size_t workspace_bytes, msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Narrow-block sparse attention ("[1/4] Add MiniMax-M3 support - #4581",
 * Kernel tuning: the QSA layers of qwen3.8-next, 12 query heads per KV head,
 * head dim 256, 4-token key blocks, timed fwd+bwd on 16k-token packs).
 * Same definition as msa_sparse_attn_fwd / _bwd with blocks of 4 tokens:
 *   q bf16 [T, Hq, 256]; k, v bf16 [T, Hkv, 256]; Hq must equal 12 Hkv;
 *   sel int32 [T, Hkv, topk], 1 <= topk <= 1024: block ids relative to the
 *   sequence start (block b = positions 4b .. 4b+3), distinct, each at most
 *   the token's own block p / 4 (larger ids set MSA_STATUS_BOUNDS and are
 *   dropped), -1 for unused slots.  A token attends to the keys j <= p of its
 *   listed blocks; the own block should be listed (a row with no key gets
 *   o = 0, lse = -inf).  max_seqlen <= 32768.
 *   o bf16 [T, Hq, 256], lse fp32 [T, Hq] (natural log);
 *   dq bf16 [T, Hq, 256], dk, dv bf16 [T, Hkv, 256].
 * Ownership, alignment, streams and errors as for the 128-token calls.
 */
MSA_API size_t msa_qsa_attn_fwd_workspace_size(int T, int S, int Hq, int Hkv, int max_seqlen);

MSA_API msa_status_t msa_qsa_attn_fwd(const void* q, const void* k, const void* v,
                              const int32_t* sel, const int32_t* cu_seqlens, int S, int T,
                              int Hq, int Hkv, int topk, int max_seqlen, float scale,
                              void* o, float* lse, void* workspace, size_t workspace_bytes,
                              msa_stream_t stream);

MSA_API size_t msa_qsa_attn_bwd_workspace_size(int T, int S, int Hq, int Hkv, int max_seqlen);

MSA_API msa_status_t msa_qsa_attn_bwd(const void* q, const void* k, const void* v,
                              const void* o, const void* dout, const float* lse,
                              const int32_t* sel, const int32_t* cu_seqlens, int S, int T,
                              int Hq, int Hkv, int topk, int max_seqlen, float scale,
                              void* dq, void* dk, void* dv, void* workspace,
                              size_t workspace_bytes, msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Decode step against a paged cache (scoring and selection rule of
 * "MiniMax-M3.1-Flash", 1 "Model Introduction", applied to one new token).
 * A page holds one 128-token block: k_cache, v_cache bf16 [num_pages, Hkv,
 * 128, 128] and kidx_cache bf16 [num_pages, Hkv, 128, 128] (index head h =
 * KV head h), post-prologue values.  block_table int32 [B, max_pages] maps
 * block c of sequence b to a page; cache_lens int32 [B] counts the cached
 * tokens INCLUDING the new one, whose position is cache_lens[b] - 1.
 * q bf16 [B, Hq, 128] and q_idx bf16 [B, Hkv, 128] are the new token's
 * post-prologue query and index query.  Per (b, h): every block up to the
 * own block is scored by its max logit, the own block plus the best 15
 * earlier ones are selected (sel_out int32 [B, Hkv, 16], may be NULL), and
 * o bf16 [B, Hq, 128] is the attention of the 16 query heads of KV head h
 * over the selected keys.
 */
MSA_API size_t msa_decode_step_workspace_size(int B, int Hq, int Hkv, int max_pages);

MSA_API msa_status_t msa_decode_step(const void* q, const void* q_idx, const void* k_cache,
                             const void* v_cache, const void* kidx_cache,
                             const int32_t* block_table, const int32_t* cache_lens, int B,
                             int Hq, int Hkv, int num_pages, int max_pages, float scale,
                             void* o, int32_t* sel_out, void* workspace,
                             size_t workspace_bytes, msa_stream_t stream);

/* msa_decode_step with the init rule of msa_index_select_ex: blocks
 * 0 .. min(n_init, own) - 1 of every sequence are always selected
 * (0 <= n_init <= 15; n_init = 0 is msa_decode_step).  Same workspace.
 */
MSA_API msa_status_t msa_decode_step_ex(const void* q, const void* q_idx, const void* k_cache,
                                const void* v_cache, const void* kidx_cache,
                                const int32_t* block_table, const int32_t* cache_lens,
                                int B, int Hq, int Hkv, int num_pages, int max_pages,
                                float scale, int n_init, void* o, int32_t* sel_out,
                                void* workspace, size_t workspace_bytes,
                                msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Decode append (the prologue of one new token per sequence, written into its
 * page; "MiniMax-M3.1-Flash", 1 "Model Introduction"; "MiniMax-M3",
 * "Architecture Notes").  Sequence b's new token is at position
 * p = cache_lens[b] - 1 (the length counts it).  q [B,Hq,128], q_idx, k, v,
 * k_idx [B,Hkv,128] are its pre-norm projections (bf16).  Then:
 *   q_out, q_idx_out = prologue(q, w_q), prologue(q_idx, w_qi) at p
 *                      (may be q / q_idx themselves, for an in-place update)
 *   k_cache[page, h, p % 128]    = prologue(k, w_k)[h]
 *   kidx_cache[page, h, p % 128] = prologue(k_idx, w_ki)[h]
 *   v_cache[page, h, p % 128]    = v[h]
 * with page = block_table[b, p / 128] and prologue = gemma norm + partial RoPE
 * as in msa_qk_norm_rope.  Caches as in msa_decode_step, which can follow on
 * the same stream.  A length outside [1, 128 max_pages] or a page outside
 * [0, num_pages) sets MSA_STATUS_BOUNDS and leaves that sequence untouched.
 */
MSA_API msa_status_t msa_decode_append(const void* q, const void* q_idx, const void* k,
                                       const void* v, const void* k_idx, const void* w_q,
                                       const void* w_qi, const void* w_k, const void* w_ki,
                                       void* k_cache, void* v_cache, void* kidx_cache,
                                       const int32_t* block_table, const int32_t* cache_lens,
                                       int B, int Hq, int Hkv, int num_pages, int max_pages,
                                       int rope_dim, float rope_base, float eps, void* q_out,
                                       void* q_idx_out, msa_stream_t stream);

/* ------------------------------------------------------------------------
 * msa_decode_step_static: the decode step above for callers that cannot
 * allocate device memory.  The pages have no counterpart of this call; it
 * exists for integration.  Some callers of a decode step own no allocator:
 * a serving engine that hands out a fixed pool of GPU memory at start-up and
 * forbids later cudaMalloc / cudaFree (which synchronize the device and
 * fragment the pool), or a plugin whose host framework gives it only the
 * tensors it computes on.  Such a caller cannot provide the workspace that
 * msa_decode_step needs.
 *
 * Same arguments, layouts and results as msa_decode_step, minus the
 * workspace: the scratch (per-block scores and per-split partial outputs)
 * lives in one fixed array in the library's device memory, sized for
 *   B * Hkv <= 256   and   max_pages <= 1024   (128K cached tokens),
 * about 9.6 MB, which every GPU that loads the library keeps until the
 * process exits.  Larger calls return MSA_ERR_UNSUPPORTED and enqueue nothing.
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.  Its first call on a device looks up that device's copy
 * of the array (a host-side query, done with the device current); make that
 * first call before any stream capture.  The address is kept per CUDA
 * context (keyed by the context's process-unique id), so after
 * cudaDeviceReset the first call in the new context looks it up again, and
 * that call too should come before any capture.  All calls share the one array, so
 * two calls whose kernels may overlap on the GPU (different streams, no
 * ordering between them) race and corrupt each other's results; calls on one
 * stream are safe.  Every scratch element a call reads is written earlier in
 * the same call, so leftovers of a previous call do not matter.
 */
MSA_API msa_status_t msa_decode_step_static(const void* q, const void* q_idx,
                                            const void* k_cache, const void* v_cache,
                                            const void* kidx_cache, const int32_t* block_table,
                                            const int32_t* cache_lens, int B, int Hq, int Hkv,
                                            int num_pages, int max_pages, float scale, void* o,
                                            int32_t* sel_out, msa_stream_t stream);

/* ------------------------------------------------------------------------
 * Launch tracing (no counterpart on the pages: measurement plumbing).
 * msa_trace_begin() clears the record and turns tracing on: from then on the
 * library brackets each of its kernel launches with a pair of CUDA events on
 * the launch stream (host-side objects, created on first use and kept).
 * msa_trace_end() waits for the recorded events, turns tracing off and writes
 * a JSON object {"<kernel>": {"launches": n, "ms": total}, ...} (NUL
 * terminated, truncated to `cap` bytes) into `json`.  Not for use inside
 * stream capture.  Tracing is process-wide and off by default.
 */
MSA_API msa_status_t msa_trace_begin(void);
MSA_API msa_status_t msa_trace_end(char* json, size_t cap);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
