/*
 * invmoe.h -- C ABI of the batch-invariant MoE layer and logprob/KL head (sm_103a).
 *
 * What the library computes (sources cited by page title and section):
 *
 *   "位级一致：前沿训练的差异化关键" (Fireworks, bit-level agreement for frontier
 *   training), section "为什么比特级一致是一个复杂的问题": a request must get the
 *   same bits whatever else shares its batch.  The router and the expert matmuls
 *   are reductions whose order must depend only on the request; the router needs
 *   a deterministic tie decision; the expert matmuls need one fixed kernel choice
 *   whatever the per-expert token count (no split-K: the page notes DeepGEMM
 *   dropped it because split-K breaks invariance).
 *
 *   "Reinforcement Learning: Why Numerical Alignment and MoE Routing Matter So
 *   Much", section "混合专家模型更难对齐": the weighted sum of expert outputs
 *   must use a pinned precision and order; k3 is the divergence metric.
 *
 *   "GLM Post-Training Beyond SFT", section "IcePop 为什么有两层 ratio": the
 *   train logprob of the exact rollout token ids, the mismatch ratio
 *   rho = exp(logp_train - logp_rollout) and the mask 1[1/beta <= rho <= beta].
 *   Section "迁移到 NPU 时": a top-k must fix ties, order, NaN handling and the
 *   index dtype.  Section "动作与概率契约": logsumexp needs comparison tests.
 *
 *   The first page, section "端到端零 KLD": the trainer follows the same
 *   bit-exact standard.  The trainer-side calls (rl_token_loss's gradient,
 *   lm_head_backward, moe_*_backward) differentiate the same definition with
 *   fixed reduction orders and no atomics.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *     The library allocates no device memory (moe_route_topk_noalloc uses one
 *     fixed array built into the library); it keeps only small host-side
 *     caches (SM count, kernel attributes).
 *   - bf16 tensors are passed as void* (raw IEEE bfloat16, row-major).
 *     float is IEEE binary32.  Index tensors are int32.
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  Arguments are validated on the
 *     host before anything is launched; on a validation error nothing is
 *     launched and the outputs are untouched.
 *   - Return value: INVMOE_OK (0) or a negative INVMOE_ERR_* code; the last
 *     error message of the calling thread is available from invmoe_last_error().
 *   - Device-side faults that the kernels detect themselves (a bounded wait that
 *     ran out) are recorded in a status word inside `workspace` and reported by
 *     invmoe_check(); the kernel that detected it stops early and its outputs
 *     are undefined.
 *   - Alignment: every tensor pointer must be 16-byte aligned.
 *   - Batch invariance: for a fixed model shape (H, E, k, F, F_shared, V) the
 *     bits of every per-token output depend only on that token's inputs, never
 *     on T, on the other tokens, or on the token's position in the batch.
 */
#ifndef INVMOE_H
#define INVMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define INVMOE_OK                       0
#define INVMOE_ERR_INVALID_ARG         -1  /* null pointer, negative size, k > E, bad beta ...   */
#define INVMOE_ERR_UNSUPPORTED_SHAPE   -2  /* a size the kernels do not tile (see each call)     */
#define INVMOE_ERR_WORKSPACE_TOO_SMALL -3  /* ws_bytes < invmoe_workspace_size(...)              */
#define INVMOE_ERR_MISALIGNED          -4  /* a pointer is not 16-byte aligned                   */
#define INVMOE_ERR_CUDA                -5  /* a CUDA runtime/driver call or a launch failed      */
#define INVMOE_ERR_DEVICE_TIMEOUT      -6  /* a kernel's bounded wait ran out (invmoe_check)     */

/* Library version (major*10000 + minor*100 + patch). */
int invmoe_version(void);

/* Message describing the last failing call made by this thread ("" if none). */
const char* invmoe_last_error(void);

/* Number of int32 elements of the dispatch plan for T tokens, E experts, top-k:
 *   plan = counts[E] | offsets[E+1] | row_token[T*k] | slot_row[T*k]
 *   counts[e]     tokens routed to expert e
 *   offsets[e]    first permuted row of expert e (offsets[0] = 0, offsets[E] = T*k);
 *                 rows of one expert are contiguous and in ascending token order
 *   row_token[r]  token whose activation sits in permuted row r
 *   slot_row[t*k + j]  permuted row holding token t's j-th ranked expert
 * The permuted row count R is exactly T*k (segments are not padded; tiles that
 * run past a segment end are masked in the kernels). */
size_t invmoe_plan_len(int T, int E, int k);

/* Bytes of device workspace that every call below accepts for these sizes
 * (F_shared = 0: no shared expert; V = 0: no head).  One workspace may be
 * reused by consecutive calls on one stream; calls that may run concurrently
 * need separate workspaces.  The first 256 bytes hold the status word; the
 * caller zero-fills the workspace once before first use. */
size_t invmoe_workspace_size(int T, int H, int E, int k, int F, int F_shared, int V);

/* Synchronise `stream`, read and clear the status word in `workspace`.
 * Returns INVMOE_OK, INVMOE_ERR_DEVICE_TIMEOUT (a kernel gave up waiting) or
 * INVMOE_ERR_INVALID_ARG (moe_route_replay was given an invalid expert index). */
int invmoe_check(void* workspace, void* stream);

/* ---------------------------------------------------------------------------
 * moe_route_topk -- router logits, top-k with lowest-index ties, gates, dispatch
 *
 *   logits[t, e] = sum_h x[t, h] * w_router[e, h]           (fp32 accumulate,
 *                  tcgen05 tile 128 x BN x 64 with BN = 64 for E <= 64, else 128,
 *                  or 64 x 64 x 64 for T <= 64; K ascending in 16-wide MMA steps,
 *                  no split-K, so a logit has the same bits whatever T)
 *   topk_idx[t, 0..k-1]: the k largest logits of row t, largest first; exact
 *                  ties (and -0 vs +0) go to the lower expert index; NaN ranks
 *                  below -inf.
 *   topk_w[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k selected
 *                  logits (softmax renormalised over the top-k, fp32, i ascending)
 *   plan         see invmoe_plan_len (deterministic counting sort; no atomics
 *                  decide any position)
 *   xp[r, :]     = x[row_token[r], :]   (bf16 copies, 16-byte vectors; each x row is read once
 *                                        and written to its k permuted rows)
 *
 * x [T, H] bf16, w_router [E, H] bf16, logits [T, E] fp32, topk_idx [T, k] int32,
 * topk_w [T, k] fp32, plan int32[invmoe_plan_len], xp [T*k, H] bf16.
 * Shapes: T >= 0, H % 64 == 0, 1 <= E <= 1024, 1 <= k <= min(E, 32).
 * ------------------------------------------------------------------------- */
int moe_route_topk(const void* x, const void* w_router, int T, int H, int E, int k,
                   float* logits, int32_t* topk_idx, float* topk_w, int32_t* plan,
                   void* xp, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_route_replay -- router replay: given expert choices, fresh gates and dispatch
 *
 * "Reinforcement Learning: Why Numerical Alignment and MoE Routing Matter So
 * Much", sections "MoE 路由会放大这种不匹配" and "Fireworks 保持训练循环一致":
 * router replay records the experts chosen during rollout and makes the trainer
 * reuse them; matching the choice is not enough, the outputs' computation and
 * combine must also match.  This call takes the recorded choices topk_idx
 * [T, k] int32 (input, not modified) instead of selecting them:
 *   logits     as moe_route_topk (same router GEMM)
 *   topk_w[t, j] = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the given
 *              experts, the sum in slot order -- bit-identical to moe_route_topk's
 *              gates when the given experts are its own choice
 *   plan, xp   as moe_route_topk, for the given experts
 * A token whose list holds an index outside [0, E) or a repeated index is
 * routed to experts 0..k-1 with NaN gates (nothing is read out of bounds) and
 * invmoe_check() then reports INVMOE_ERR_INVALID_ARG.
 * Workspace: invmoe_workspace_size(T, H, E, k, ...) bytes.
 * ------------------------------------------------------------------------- */
int moe_route_replay(const void* x, const void* w_router, const int32_t* topk_idx, int T, int H, int E, int k,
                     float* logits, float* topk_w, int32_t* plan, void* xp,
                     void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_grouped_ffn -- grouped SwiGLU expert GEMMs (+ optional shared expert)
 *
 * For every expert e and each of its permuted rows r in [offsets[e], offsets[e+1]):
 *   g = xp[r] . Wg_e^T,  u = xp[r] . Wu_e^T      (fp32 in TMEM, K ascending)
 *   h[r, f] = bf16_rne( silu(g_f) * u_f ),  silu(g) = g / (1 + exp(-g))  (fp32)
 *   y[r, :] = h[r] . W2_e^T                       (fp32 accumulate, stored fp32)
 * One tile shape (128 rows x 256 columns x 64 K) for every expert whatever its
 * row count; K is always walked in ascending order; no split-K.
 * Shared expert (F_shared > 0): the same two GEMMs over all T tokens of
 * x_shared with ws13/ws2, result in y_shared [T, H] fp32.
 *
 * xp [T*k, H] bf16, plan from moe_route_topk, w13 [E, 2F, H] bf16 (rows 0..F-1
 * gate, F..2F-1 up), w2 [E, H, F] bf16, h [T*k, F] bf16, y [T*k, H] fp32,
 * x_shared [T, H] bf16, ws13 [2*F_shared, H] bf16, ws2 [H, F_shared] bf16.
 * Shapes: H % 64 == 0, F % 128 == 0, F_shared % 128 == 0.
 * ------------------------------------------------------------------------- */
int moe_grouped_ffn(const void* xp, const int32_t* plan, const void* w13, const void* w2,
                    int T, int H, int E, int k, int F, void* h, float* y,
                    const void* x_shared, const void* ws13, const void* ws2, int F_shared,
                    float* y_shared, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_combine -- fp32 fixed-order weighted combine
 *
 *   out[t, :] = ((w[t,0]*y[slot_row[t,0]] + w[t,1]*y[slot_row[t,1]]) + ...)
 *               + y_shared[t]      (if y_shared != NULL)
 * in fp32, slots in rank order j = 0..k-1, every product and sum rounded
 * separately (no fused multiply-add), shared expert added last.
 * out_bf16 (nullable) receives bf16_rne(out).
 * y [T*k, H] fp32, topk_w [T, k] fp32, plan from moe_route_topk, out [T, H] fp32.
 * Shapes: H % 4 == 0.
 * ------------------------------------------------------------------------- */
int moe_combine(const float* y, const float* topk_w, const int32_t* plan, const float* y_shared,
                int T, int H, int E, int k, float* out, void* out_bf16, void* stream);

/* ---------------------------------------------------------------------------
 * moe_layer_forward -- the whole layer in one call
 *
 * moe_route_topk, then moe_grouped_ffn (with the shared expert on x when
 * F_shared > 0), then moe_combine: exactly those three calls' kernels (so the
 * same bits), for callers that serve one small batch at a time and want one
 * host call per layer.  Arguments, layouts and errors as the three calls;
 * ws13, ws2 and y_shared are ignored when F_shared == 0; the workspace is
 * invmoe_workspace_size(T, H, E, k, F, F_shared, 0) bytes.
 * With a shared expert, at most 1024 tokens (see invmoe_shared_overlap) and a
 * workspace of that size, the shared expert's two GEMMs run on a stream of the
 * library's own (one per device, created on the first such call that is not
 * made during a graph capture) while the routing and the routed experts run on
 * `stream`; `stream` waits for that stream (an event) before the combine, so on
 * return the call is ordered on `stream` as if it had run there alone, and a
 * graph captured from `stream` holds both branches.  Such calls from several
 * host threads are serialised by a lock around their launches.
 * ------------------------------------------------------------------------- */
int moe_layer_forward(const void* x, const void* w_router, const void* w13, const void* w2,
                      const void* ws13, const void* ws2, int T, int H, int E, int k, int F, int F_shared,
                      float* logits, int32_t* topk_idx, float* topk_w, int32_t* plan, void* xp, void* h,
                      float* y, float* y_shared, float* out, void* out_bf16, void* workspace,
                      size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * lm_logprob_kl -- vocab projection, chunked two-pass log-sum-exp, logprob, k3, IcePop
 *
 *   z[t, v] = sum_h hidden[t, h] * w_vocab[v, h]     (fp32 in TMEM, tcgen05 tile 128 x 256 x 64)
 *   pass 1, in the projection's epilogue, chunk c = columns [256c, 256c+256):
 *           m_c = max z;  s_c = sum of exp(z - m_c): column j of the chunk is added,
 *           in ascending j, to accumulator j mod 8, then s_c = ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7))
 *   pass 2, partials folded as (M, S) + (m, s) = (M', S*exp(M - M') + s*exp(m - M')),
 *           M' = max(M, m), in a fixed order: lane l of a warp folds chunks
 *           [l*P, (l+1)*P), P = ceil(V/256/32), in ascending order, then the 32 lane
 *           results fold by a xor butterfly (16, 8, 4, 2, 1);  lse = M + log(S)
 *   logp[t] = z[t, target[t]] - lse[t]
 *   if rollout_logp != NULL:
 *     d = logp - rollout_logp;  k3 = expm1(d) - d;  rho = exp(d);
 *     mask = (1/beta <= rho) && (rho <= beta)      (all fp32)
 * A target outside [0, V) yields logp = NaN for that token.
 *
 * hidden [T, H] bf16, w_vocab [V, H] bf16, target [T] int32, rollout_logp [T]
 * fp32 (nullable: k3/mask not written), logits [T, V] fp32 (nullable: the logits
 * are then never written to memory), logp [T] fp32, lse/k3 [T] fp32 and mask [T]
 * uint8 (nullable).
 * Shapes: H % 64 == 0, V % 4 == 0, beta >= 1.
 * With fewer than 64 tokens and a workspace of invmoe_workspace_size(T, H, ...,
 * V) bytes, the hidden rows are first copied into the workspace, padded to 64
 * rows (faster tiles; the rows past T are never stored, the results are the
 * same); a workspace large enough for the partials alone also works.
 * ------------------------------------------------------------------------- */
int lm_logprob_kl(const void* hidden, const void* w_vocab, const int32_t* target,
                  const float* rollout_logp, int T, int H, int V, float beta,
                  float* logits, float* logp, float* lse, float* k3, uint8_t* mask,
                  void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Vocabulary-parallel head: lm_logprob_partials on each vocabulary shard, then
 * lm_logprob_merge over the gathered partials.
 *
 * "GLM Post-Training Beyond SFT", section "动作与概率契约": the log-sum-exp over
 * a vocabulary split across devices needs comparison tests; "位级一致：前沿训练
 * 的差异化关键", section "为什么比特级一致是一个复杂的问题": a cross-device
 * reduction must not change its order with the size of the job.  Here the
 * vocabulary is cut at 256-column chunk boundaries, every shard computes pass 1
 * of the log-sum-exp for its own chunks with the same tile and K order as
 * lm_logprob_kl, and pass 2 folds the chunks in the same fixed global order as
 * lm_logprob_kl -- so any split into shards gives the bits of the unsharded
 * call.  lm_logprob_kl is exactly these two calls over one shard [0, V).
 * ------------------------------------------------------------------------- */

/* Pass 1 on the vocabulary shard [v0, v1): for each token t and each chunk
 * c = v0/256 + j of the shard (columns [256c, 256c + 256) of the whole
 * vocabulary, clipped to v1):
 *   partials[2 * (t * ld_part + j)]     = m = max z[t, chunk]
 *   partials[2 * (t * ld_part + j) + 1] = s = sum exp(z - m)   (the lm_logprob_kl order)
 * and, for tokens whose target lies in [v0, v1), tgt_logit[t] = z[t, target[t]]
 * (other tokens' entries are not written).
 *
 * hidden [T, H] bf16; w_vocab_shard = rows [v0, v1) of the vocabulary projection,
 * [v1 - v0, H] bf16; target [T] int32 (ids in the whole vocabulary); logits
 * (nullable) = the whole [T, V] fp32 logits array, of which columns [v0, v1) are
 * written; partials (8-byte aligned) as above, ld_part >= the shard's chunk count
 * (in (m, s) pairs); tgt_logit [T] fp32.  workspace: at least 256 bytes (status).
 * Shapes: H % 64 == 0, V % 4 == 0, 0 <= v0 < v1 <= V, v0 % 256 == 0, and
 * v1 % 256 == 0 unless v1 == V. */
int lm_logprob_partials(const void* hidden, const void* w_vocab_shard, const int32_t* target,
                        int T, int H, int V, int v0, int v1, float* logits, float* partials,
                        long long ld_part, float* tgt_logit, void* workspace, size_t ws_bytes,
                        void* stream);

/* Pass 2 and the per-token outputs (as lm_logprob_kl) from partials laid out in
 * shards of shard_chunks chunks: the (m, s) pair of global chunk c of token t is at
 *   partials + 2 * ((c / shard_chunks) * shard_stride + t * ld_part + c % shard_chunks)
 * and token t's target logit at tgt_logit[(target[t] / 256 / shard_chunks) * tgt_stride + t]
 * (read from the shard that owns the target; nothing is summed across shards).
 * One [T, NCH] array (NCH = ceil(V / 256)): shard_chunks = ld_part = NCH,
 * shard_stride = tgt_stride = 0.  An all-gather of n shards' [T, P] partials into
 * [n][T][P] and of their [T] target logits into [n][T]: shard_chunks = ld_part = P,
 * shard_stride = T * P, tgt_stride = T (the last shard may hold fewer than P
 * chunks; unused entries are not read).  Other arguments and outputs as
 * lm_logprob_kl. */
int lm_logprob_merge(const float* partials, long long ld_part, int shard_chunks, long long shard_stride,
                     const float* tgt_logit, long long tgt_stride, const int32_t* target,
                     const float* rollout_logp, int T, int V, float beta, float* logp, float* lse,
                     float* k3, uint8_t* mask, void* stream);

/* ---------------------------------------------------------------------------
 * Expert-parallel layer: the experts split over ranks, each rank owning the
 * contiguous range [e0, e1) (E_local = e1 - e0 experts).
 *
 * Every rank routes its own tokens with the whole router (moe_route_topk).
 * Its xp rows are sorted by expert, so the rows for the owner of [e0, e1) are
 * the one slice xp[offsets[e0] : offsets[e1]); an all-to-all (the caller's
 * collective) delivers to each owner the rows of every source, source-major.
 * The owner regroups them expert-major (moe_ep_regroup), runs its experts with
 * moe_grouped_ffn (T = R received rows, k = 1, E = E_local, plan = plan_local,
 * w13/w2 = its experts' weights), puts the output rows back in the received
 * order (moe_ep_ungroup) and returns them with the reverse all-to-all; each
 * source then holds y in its own xp order and combines locally (moe_combine),
 * adding the shared expert it computed itself (moe_shared_expert).
 * Rows are only moved between devices, never reduced across them, and an
 * expert output row depends on its own input row only (one fixed tile, K
 * ascending), so every output has the bits of the one-device layer
 * ("位级一致：前沿训练的差异化关键", section "为什么比特级一致是一个复杂的问题").
 * ------------------------------------------------------------------------- */

/* recv_xp [R, H] bf16: the received rows, source-major (source 0's rows for
 * local experts 0, 1, ..., then source 1's, ...; within one (source, expert) in
 * the source's order); recv_counts [n_src, E_local] int32 (device): rows that
 * source s sent for local expert e.  Outputs: xp_local [R, H] bf16 (expert-major;
 * within an expert, sources ascending), plan_local int32 [2 * E_local + 1] =
 * counts[E_local] | offsets[E_local + 1] (the plan moe_grouped_ffn reads), and
 * row_src [R] int32: the received row each xp_local row was copied from.
 * If the counts do not add up to R, no access goes out of bounds, the status
 * word records it and invmoe_check() returns INVMOE_ERR_INVALID_ARG.
 * workspace: at least 256 bytes (status).  Shapes: H % 8 == 0,
 * E_local <= 1024, n_src * E_local <= 65535. */
int moe_ep_regroup(const void* recv_xp, const int32_t* recv_counts, int n_src, int E_local, int R, int H,
                   void* xp_local, int32_t* plan_local, int32_t* row_src, void* workspace,
                   size_t ws_bytes, void* stream);

/* y_send[row_src[i], :] = y_local[i, :] for i < R: the expert outputs back in
 * the received (source-major) order.  y_local, y_send [R, H] fp32, row_src from
 * moe_ep_regroup.  Shapes: H % 4 == 0. */
int moe_ep_ungroup(const float* y_local, const int32_t* row_src, int R, int H, float* y_send, void* stream);

/* The shared expert alone (as inside moe_grouped_ffn): y_shared [T, H] fp32 =
 * SwiGLU(x) with ws13 [2 * F_shared, H], ws2 [H, F_shared] bf16, on the CTA-pair
 * engine; the bf16 hidden activation lives in the workspace
 * (invmoe_workspace_size(T, H, 0, 0, 0, F_shared, 0) bytes).
 * Shapes: H % 64 == 0, F_shared % 128 == 0. */
int moe_shared_expert(const void* x, const void* ws13, const void* ws2, int T, int H, int F_shared,
                      float* y_shared, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_route_topk_noalloc -- moe_route_topk for callers that cannot allocate
 *
 * The source pages have no counterpart of this call; it exists for callers that
 * may not allocate device memory where they route tokens (a serving loop under a
 * fixed memory budget, where cudaMalloc could fail or stall the device, or a
 * plain-C host that only holds the buffers it was given).  It computes exactly
 * what moe_route_topk computes, with the same kernels, but takes no workspace:
 * its scratch (status word, schedule counter, per-chunk expert counts) is one
 * fixed array of 1 MiB + 256 bytes inside the library, held by every GPU that
 * loads the library until the process exits.
 *   - Limit: ceil(T/64) * E <= 262144 (for example T <= 65536 at E = 256);
 *     larger sizes return INVMOE_ERR_UNSUPPORTED_SHAPE and launch nothing.
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 *   - The first call on each device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *     The address is kept for the life of the process: it does not survive a
 *     cudaDeviceReset() (or anything else that replaces the device's primary
 *     context), after which this call must not be used in that process.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (the status word is cleared at the start of every call): calls
 *     that overlap on the GPU (other streams, other host threads) race.
 *   - status (nullable, 4-byte aligned device pointer, caller-owned): receives
 *     the call's status word (non-zero = a bounded device wait ran out).
 * Other arguments, layouts and errors: as moe_route_topk.
 * ------------------------------------------------------------------------- */
int moe_route_topk_noalloc(const void* x, const void* w_router, int T, int H, int E, int k,
                           float* logits, int32_t* topk_idx, float* topk_w, int32_t* plan,
                           void* xp, unsigned int* status, void* stream);

/* ---------------------------------------------------------------------------
 * lm_head_backward -- deterministic backward of the vocabulary projection
 *
 * The trainer's side of the same definition ("位级一致：前沿训练的差异化关键",
 * section "端到端零 KLD": the trainer follows the same bit-exact standard as the
 * serving path).  For the per-token loss L = sum_t g[t] * logp[t] (g = dL/dlogp,
 * e.g. rl_token_loss's grad_logp; g[t] = 0 for a token the IcePop mask drops):
 *   z[t, v]   recomputed exactly as lm_logprob_kl computes it (same tile, same
 *             K order, so bit-identical)
 *   dz[t, v]  = bf16_rne( g[t] * (onehot(v == target[t]) - exp(z[t, v] - lse[t])) )
 *             fp32: p = exp(z - lse); 1 - p at the target column, -p elsewhere;
 *             one fp32 multiply by g[t]; then rounded to bf16
 *   d_hidden[t, h] = sum_v dz[t, v] * w_vocab[v, h]       v ascending in 64-wide blocks
 *   d_wvocab[v, h] = sum_t dz[t, v] * hidden[t, h]        t ascending in 64-wide blocks
 * Each output element is produced by one CTA pair that walks its reduction in
 * the same order on every call (no split reduction, no atomics), so repeated
 * calls give identical bits whatever the schedule; a row of d_hidden depends on
 * its own token only (batch-invariant), as in the forward.
 *
 * hidden [T, H] bf16, w_vocab [V, H] bf16, target [T] int32 (in [0, V)), lse [T]
 * fp32 (from lm_logprob_kl), grad_logp [T] fp32; outputs (device, caller-owned):
 * dlogits [T, V] bf16, d_hidden [T, H] fp32 (nullable: not computed),
 * d_wvocab [V, H] fp32 (nullable: not computed).  All 16-byte aligned.
 * workspace: invmoe_workspace_size(T, H, 0, 0, 0, 0, V) bytes suffice (only the
 * status block is used).
 * Shapes: H % 64 == 0, V % 8 == 0.  T may be any size >= 0.
 * ------------------------------------------------------------------------- */
int lm_head_backward(const void* hidden, const void* w_vocab, const int32_t* target, const float* lse,
                     const float* grad_logp, int T, int H, int V, void* dlogits, float* d_hidden,
                     float* d_wvocab, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * MoE layer backward: moe_combine_backward, then moe_grouped_ffn_backward, then
 * moe_route_backward.
 *
 * The trainer's side of the same definition ("位级一致：前沿训练的差异化关键",
 * section "端到端零 KLD").  For the upstream gradient dout [T, H] fp32 of the
 * layer output, with the forward's routing (topk_idx, topk_w, plan), permuted
 * rows xp and per-slot expert outputs y:
 *   dgate[t,j] = <dout[t], y[slot_row[t,j]]>;  dy[slot_row[t,j]] = bf16(topk_w[t,j] * dout[t])
 *   expert e, on its rows:  dh = dy W2_e;  g, u recomputed (the forward's tile
 *     and K order); dg = (dh*u) * s(1 + g(1 - s)), du = dh * silu(g), s = sigmoid(g),
 *     [dg | du] rounded to bf16 (the forward's h is taken as silu(g)*u: its bf16
 *     rounding is not differentiated);  dxp = [dg | du] W13_e;
 *     dW2_e = dy^T h,  dW13_e = [dg | du]^T xp, over the expert's rows only
 *   shared expert: the same with dy = bf16(dout) and x
 *   router: ds_j = w_j (dgate_j - sum_i w_i dgate_i) at column topk_idx[t,j] of
 *     dlogits [T, E] (bf16, 0 elsewhere);  dx_router = dlogits W_router,
 *     dW_router = dlogits^T x
 *   dx[t] = ((sum_j dxp[slot_row[t,j]]) + dx_shared[t]) + dx_router[t]  (slots in rank order)
 * Every output element is reduced in one fixed order by one CTA (no split
 * reduction, no atomics): repeated calls give identical bits, and dx rows and
 * the per-slot rows depend on their own token only (batch-invariant); the
 * weight gradients are sums over the batch by definition.
 * ------------------------------------------------------------------------- */

/* Workspace for moe_grouped_ffn_backward and moe_route_backward: status block,
 * then (each part 256-byte aligned) dh [T*k, F] fp32, [dg | du] [T*k, 2F] bf16,
 * recomputed h [T*k, F] bf16, the same three for the shared expert ([T, F_shared],
 * [T, 2*F_shared], [T, F_shared]) and dlogits [T, E] bf16.  After a call those
 * parts hold that call's intermediate results. */
size_t invmoe_backward_workspace_size(int T, int H, int E, int k, int F, int F_shared);

/* dout [T, H] fp32, y [T*k, H] fp32 (the forward's per-slot outputs), topk_w
 * [T, k] fp32, plan from the forward; outputs dy [T*k, H] bf16 (permuted rows, as
 * xp), dgate [T, k] fp32, dout_bf16 [T, H] bf16 (nullable: the shared expert's
 * operand).  dgate: lane l of the slot's warp adds elements 4(l + 32i) .. +3 in
 * ascending order, then a xor butterfly.  Shapes: H % 4 == 0, k <= 32. */
int moe_combine_backward(const float* dout, const float* y, const float* topk_w, const int32_t* plan,
                         int T, int H, int E, int k, void* dy, float* dgate, void* dout_bf16, void* stream);

/* xp [T*k, H] bf16, plan, w13 [E, 2F, H] bf16, w2 [E, H, F] bf16, dy [T*k, H] bf16;
 * outputs dxp [T*k, H] fp32, dw13 [E, 2F, H] fp32 and dw2 [E, H, F] fp32 (both
 * nullable: not computed).  Shared expert (F_shared > 0): x_shared [T, H] bf16,
 * ws13 [2*F_shared, H], ws2 [H, F_shared] bf16, dout_bf16 [T, H] bf16; outputs
 * dx_shared [T, H] fp32, dws13 [2*F_shared, H] and dws2 [H, F_shared] fp32
 * (nullable).  An expert no token chose gets zero weight gradients.
 * Shapes: H % 64 == 0, F % 128 == 0, F_shared % 128 == 0, E <= 1024. */
int moe_grouped_ffn_backward(const void* xp, const int32_t* plan, const void* w13, const void* w2,
                             const void* dy, int T, int H, int E, int k, int F, float* dxp, float* dw13,
                             float* dw2, const void* x_shared, const void* ws13, const void* ws2,
                             const void* dout_bf16, int F_shared, float* dx_shared, float* dws13,
                             float* dws2, void* workspace, size_t ws_bytes, void* stream);

/* x [T, H] bf16, w_router [E, H] bf16, topk_idx [T, k] int32, topk_w [T, k] fp32,
 * dgate [T, k] fp32, dxp [T*k, H] fp32, plan, dx_shared [T, H] fp32 (nullable);
 * outputs dx [T, H] fp32 (the layer input's gradient) and dw_router [E, H] fp32
 * (nullable).  Shapes: H % 64 == 0, E % 8 == 0, k <= 32. */
int moe_route_backward(const void* x, const void* w_router, const int32_t* topk_idx, const float* topk_w,
                       const float* dgate, const float* dxp, const int32_t* plan, const float* dx_shared,
                       int T, int H, int E, int k, float* dx, float* dw_router, void* workspace,
                       size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * rl_token_loss -- IcePop-masked clipped policy loss and DIS weights per token
 *
 * "GLM Post-Training Beyond SFT", sections "GRPO 在优化什么" (clipped objective
 * min(r A, clip(r, 1-eps_l, 1+eps_h) A), eps_l = 0.2, eps_h = 0.28),
 * "IcePop 为什么有两层 ratio" (the trust mask multiplies the token loss) and
 * "Direct Double-Sided Importance Sampling" (f(r) = r inside (1-eps_l, 1+eps_h),
 * else 0).  Per token, fp32:
 *   rho = exp(logp_train - logp_rollout);  r = exp(logp_train - logp_old)
 *   icepop_mask = 1/beta <= rho <= beta
 *   loss = icepop_mask ? -min(r*A, clip(r, 1-eps_low, 1+eps_high)*A) : 0
 *   dis_weight = (1-eps_low < rho < 1+eps_high) ? rho : 0
 * loss_mean (nullable, [1]) = sum(loss) / T in a fixed order (one block: thread i
 * adds elements i, i+1024, ... ascending, then xor butterflies inside and across
 * warps).  logp_old nullable (then r = rho); icepop_mask, dis_weight nullable.
 * grad_logp (nullable) = d loss_mean / d logp_train, the mask held fixed:
 *   icepop_mask && r*A <= clip(r)*A ? -(r*A) / T : 0
 * (the unclipped term is the minimum, which holds for every r inside the clip
 * window; where the clipped term is strictly smaller it is constant in r).
 * All [T] device arrays; fp32 except icepop_mask (uint8).
 * ------------------------------------------------------------------------- */
int rl_token_loss(const float* logp_train, const float* logp_old, const float* logp_rollout,
                  const float* advantage, int T, float beta, float eps_low, float eps_high,
                  uint8_t* icepop_mask, float* dis_weight, float* loss, float* loss_mean,
                  float* grad_logp, void* stream);

/* ---------------------------------------------------------------------------
 * Diagnostics
 * ------------------------------------------------------------------------- */

/* d[m, n] = sum_k a[m, k] * b[n, k] (fp32 out, ldd = N): the dense tcgen05 GEMM
 * engine on its own, used by the tests to check the engine at ragged sizes.
 * variant selects the tile configuration the other calls use:
 *   0 = 128 x 256 tile, one row tile per unit
 *   1 = 128 x 256 tile, two row tiles per unit (vocab and expert down projections)
 *   2 = 128 x 128 tile, 3 = 128 x 64 tile (router logits for E <= 128 / 64)
 *   4 = 256 x 256 tile computed by a CTA pair (cta_group::2) on two SMs
 *   5 = as 4 with b MN-major: b is [K, N] (d = a * b), K % 8 == 0, N % 8 == 0
 *   6 = as 4 with a and b MN-major: a is [K, M], b is [K, N] (d = a^T * b),
 *       any K >= 1, M % 8 == 0, N % 8 == 0
 * plus 256 to order the work units column-block-major (the vocab projection's order).
 * a [M, K] bf16, b [N, K] bf16 unless stated.  Shapes (0..4): K % 64 == 0, N % 4 == 0. */
int invmoe_gemm_bf16(const void* a, const void* b, int M, int N, int K, float* d, int variant,
                     void* workspace, size_t ws_bytes, void* stream);

/* Per-kernel timing.  While enabled, every kernel launch made by this library
 * is bracketed by a pair of CUDA events recorded on the launch stream (events
 * come from a host-side pool; no device memory is allocated).
 * invmoe_profile_collect() waits for the recorded events, writes up to
 * max_entries aggregated rows -- kernel name (NUL-terminated, at most 47 chars,
 * in a 48-byte slot of `names`), total milliseconds and launch count -- drops
 * the records and returns the number of rows (negative on error). */
int invmoe_profile_enable(int on);
int invmoe_profile_collect(char* names, float* total_ms, int* launches, int max_entries);

/* Programmatic dependent launch (on by default): every kernel of this library is
 * launched so that it may be scheduled while the previous kernel on its stream is
 * still finishing; it runs only its set-up (shared memory, TMEM, descriptor
 * prefetch) before waiting for that kernel to complete, so results are the same
 * either way.  invmoe_pdl_enable(0) launches them plainly (for timing
 * comparisons); the setting applies to calls made after it. */
int invmoe_pdl_enable(int on);

/* Where moe_layer_forward runs the shared expert (calls made after it): 0 on
 * `stream` after the routed experts, 1 on the library's side stream beside the
 * routing and the routed experts, 2 (default) the side stream for batches of at
 * most 1024 tokens.  The kernels and their results are the same either way. */
int invmoe_shared_overlap(int mode);

/* Engine of moe_grouped_ffn's two routed-expert GEMMs (calls made after it):
 * 0 puts each expert's tokens on the MMA's M side in 128-row tiles (64 for a
 * last tile of at most 64 rows); 1 puts its weight rows on the M side and its
 * tokens on the N side (any multiple of 16 tokens, on a CTA pair, in units of
 * at most 64 tokens for batches of at most 1024 slots or 16 per expert, 128 for
 * at most 64 per expert, else 320); 2 (default) takes 1 for the gate/up GEMM,
 * and for the down projection 1 when the batch holds at most 8 slots and
 * H > 1024 (one decode token of a wide layer) or, with F >= 2048, averages at
 * most 64 or at least 256 slots per expert, else 0.  Both walk every element's
 * reduction in the same order and give the same bits (tested), so the choice
 * never changes an output. */
int invmoe_expert_engine(int which);

/* Launch a one-CTA kernel that waits on an mbarrier nothing ever completes,
 * with a wait limit of `timeout_us` microseconds (1..2000000).  The kernel
 * gives up, records INVMOE_ERR_DEVICE_TIMEOUT in the status word and returns;
 * invmoe_check() must then report it.  Exercises the timeout path without
 * hanging or faulting the GPU. */
int invmoe_debug_timeout_probe(void* workspace, size_t ws_bytes, int timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* INVMOE_H */
