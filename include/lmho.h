/*
 * lmho.h -- C ABI of the GB300 (sm_103a) LM-head loss library.
 *
 * The operations are the four contracts of the KernelIndex operation pages
 * "Cross-entropy loss", "Vocab-parallel cross-entropy, Megatron layout",
 * "Fused linear + CPO loss" (its cross-entropy core) and "Fused linear + JSD".
 * The pages give tensor names, dtypes and shapes (section "Semantics") and
 * name the losses; the arithmetic is the textbook definition of each name:
 *
 *   cross-entropy of row i:  loss_i = ln(sum_v exp(z_iv)) - z_{i, t_i}
 *   generalized JSD:         JSD_b(P||Q) = b KL(P||M) + (1-b) KL(Q||M),
 *                            M = b P + (1-b) Q, natural log.
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers, owned by the caller, contiguous and
 *     row-major.  bf16 tensors are passed as their 16-bit patterns
 *     (const uint16_t*), so this header needs no CUDA include.  Exception: the
 *     CE row calls (ce_fwd_f32, ce_fwd_sbv_bf16, ce_partials_sbv_bf16,
 *     ce_partials_f32) also take logits and targets in pinned (page-locked,
 *     mapped) host memory: their kernels then read them over the host link
 *     (one streaming read, at the link's rate; the results are the same bits
 *     as from device memory).  Outputs and workspaces are always device
 *     memory.  lmho_copy_h2d, the transfer utility, reads pinned host memory
 *     too.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work on it: they never synchronise, never allocate and
 *     keep no state between calls.  They are thread-safe.  The exceptions are
 *     the process-wide tuning settings at the end of this header
 *     (lmho_set_ce_variant, lmho_set_raster_group, lmho_set_wait_timeout_ns):
 *     a change made by one thread applies to later calls of every thread.
 *     They choose kernels and limits, never results beyond rounding.  The
 *     measurement hook lmho_set_launch_events is per host thread.
 *   - Programmatic dependent launch: the cross-entropy forward row kernels
 *     are launched as programmatic dependents of the kernel before them on
 *     the stream and wait for that kernel's completion before touching
 *     memory, so they are correct after any producer.  They, and the short-row
 *     forward + backward kernel, also let the next kernel on the stream launch
 *     early: a caller's kernel launched with programmatic stream serialization
 *     must wait (griddepcontrol.wait) before it reads a call's outputs, as that
 *     launch mode requires of any dependent.
 *   - "No mutation or aliasing" (every page, section Semantics): inputs are
 *     never written, and an output or workspace byte range that overlaps an
 *     input (or each other) is rejected with LMHO_ERR_ALIAS.
 *   - Host-checkable errors (NULL pointer, a size <= 0, aliasing, a short
 *     workspace, a device that is not compute capability 10.3, an unsupported
 *     hidden size) return a status and launch nothing.  Targets live on the
 *     device and are not checked on the host: a target outside [0, V) makes
 *     that token's loss NaN, and a mean over it NaN.
 *   - NaN logits propagate (the token's loss is NaN); a +inf logit gives NaN.
 *   - Results are bitwise reproducible run to run (fixed-order reductions).
 *   - Workspaces are caller-owned device memory, 256-byte aligned, and must be
 *     ZERO-FILLED before their first use; every call leaves the words that
 *     must start at zero back at zero.  One workspace serves one call at a
 *     time: calls in flight at once need distinct workspaces.
 */
#ifndef LMHO_H_
#define LMHO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LMHO_OK = 0,
  LMHO_ERR_INVALID_ARG = 1,  /* NULL pointer, size <= 0, bad option            */
  LMHO_ERR_ALIAS = 2,        /* an output/workspace range overlaps another    */
  LMHO_ERR_WORKSPACE = 3,    /* ws_bytes below the *_workspace_bytes() value  */
  LMHO_ERR_UNSUPPORTED = 4,  /* not an sm_103 device, or H % 8 != 0           */
  LMHO_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch, attribute)*/
  LMHO_ERR_TIMEOUT = 6       /* a bounded in-kernel wait gave up (device side)*/
} lmho_status;

/* Human-readable text of a status code (static storage, never NULL). */
const char* lmho_strerror(int status);

/* Library version, major*10000 + minor*100 + patch. */
int lmho_version(void);

/* ------------------------------------------------------------------------
 * Flat cross-entropy, fp32 logits, mean-reduced.
 * Page "Cross-entropy loss", section Semantics: logits float [tokens, vocab],
 * target int64 [tokens], loss float [1].
 *
 *   logits  [T, V] fp32 device, row i at logits + i*V (any 4-byte alignment;
 *           rows whose start is not 16-byte aligned are peeled in-kernel)
 *   target  [T] int64 device
 *   loss    [1] fp32 device output: (1/T) sum_i loss_i
 *   ws      device workspace of ws_bytes >= ce_workspace_bytes(T, V), zeroed
 *           before first use.  After the call completes, the first T floats
 *           of ws hold the per-token losses loss_i.
 * Two kernel launches: the row kernel, then a one-block mean kernel launched
 * as its programmatic dependent (it starts while the rows drain and waits
 * in-kernel for their completion); the mean's summation order is fixed.
 * ------------------------------------------------------------------------ */
size_t ce_workspace_bytes(int64_t T, int64_t V);
int ce_fwd_f32(const float* logits, const int64_t* target, int64_t T, int64_t V,
               float* loss, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * ce_fwd_f32 without a caller workspace, for callers that cannot allocate
 * device memory: a process that reserved its device-memory pool up front and
 * must not grow its footprint, a plug-in running inside another framework's
 * allocator, a binding with no device allocator to hand.  The operation pages
 * have no counterpart of this entry point: it is a library convenience.
 *
 * Same operation, arguments, result and kernels as ce_fwd_f32, except that
 * the per-token losses and the control words live in a scratch array inside
 * the library: a file-scope __device__ array of 256 KB + 256 bytes that every
 * GPU which loads the library holds until the process exits.
 *   - T is limited to 65536 tokens; larger T returns LMHO_ERR_INVALID_ARG.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating routine.
 *   - The first call on a device (and the first after that device's context
 *     has been replaced, e.g. by cudaDeviceReset) looks up the array's device
 *     address with that device current and caches it; make that first call
 *     before any stream capture on that device.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; each call first clears the control words it needs at
 *     zero (one cudaMemsetAsync on `stream`, then the kernels).  Calls that
 *     overlap on the GPU (other streams, other threads) race on the array and
 *     give undefined results: serialise them.
 * ------------------------------------------------------------------------ */
int ce_fwd_f32_noalloc(const float* logits, const int64_t* target, int64_t T, int64_t V,
                       float* loss, void* stream);

/* ------------------------------------------------------------------------
 * Megatron-layout cross-entropy, bf16 logits, per-token fp32 losses.
 * Page "Vocab-parallel cross-entropy, Megatron layout", summary (bf16 logits,
 * per-token fp32 losses, tensor parallel size 1) and section Semantics:
 * logits [seq, batch, vocab], target int64 [seq, batch], loss fp32 [seq, batch].
 *
 *   logits  [S, B, V] bf16 device (row s*B+b at logits + (s*B+b)*V)
 *   target  [S, B] int64 device
 *   loss    [S, B] fp32 device output, loss[s*B+b] = loss of that token;
 *           accumulation is fp32.
 * No workspace.  One kernel launch.
 * ------------------------------------------------------------------------ */
int ce_fwd_sbv_bf16(const uint16_t* logits, const int64_t* target, int64_t S, int64_t B,
                    int64_t V, float* loss, void* stream);

/* ------------------------------------------------------------------------
 * Vocab-parallel (tensor-parallel) Megatron-layout cross-entropy.
 * Page "Vocab-parallel cross-entropy, Megatron layout", summary: with the
 * vocabulary sharded over tensor-parallel ranks each rank holds only its own
 * vocab range, so the local logits are [seq, batch, V_local].  A rank reduces
 * each token to its shard's partial; the ranks exchange the partials (one
 * all-gather of 12 bytes per token per rank, done by the caller, e.g. NCCL);
 * every rank then merges all shards into the per-token losses.
 *
 * ce_partials_sbv_bf16: one shard.
 *   logits_local [S, B, V_local] bf16 device: global vocab columns
 *                [vocab_start, vocab_start + V_local) of every token
 *   target       [S, B] int64 device, GLOBAL vocab indices
 *   partials     [3][S*B] fp32 device output: m[i] = max of the shard's
 *                logits of token i, s[i] = sum of exp(z - m[i]) over the
 *                shard, z[i] = the target logit when the target lies in this
 *                shard, else -inf.  (Token i = s*B + b.)
 *   vocab_start >= 0.  One kernel launch (the Megatron CE row decompositions).
 *
 * ce_merge_partials: `shards` blocks of partials, contiguous in shard order
 * ([shards][3][S*B] fp32 device, as an all-gather of the per-rank blocks in
 * rank order leaves them), merged per token in that order:
 *   M = max m_j,  loss = M + ln(sum_j s_j exp(m_j - M)) - max_j z_j;
 *   target [S, B] int64 device (global), V = the global vocabulary size; the
 *   shards must cover [0, V) exactly once (not checked).  A target outside
 *   [0, V) gives NaN.  loss [S, B] fp32 device output.  One kernel launch.
 * Both: no workspace; accumulation in fp32; outputs must not overlap inputs.
 * ------------------------------------------------------------------------ */
int ce_partials_sbv_bf16(const uint16_t* logits_local, const int64_t* target, int64_t S,
                         int64_t B, int64_t V_local, int64_t vocab_start, float* partials,
                         void* stream);
int ce_merge_partials(const float* partials, int64_t shards, const int64_t* target, int64_t S,
                      int64_t B, int64_t V, float* loss, void* stream);

/* ce_partials_f32: the same shard partials for the flat fp32 layout (page
 * "Cross-entropy loss", logits [tokens, vocab]) with the vocabulary split the
 * same way: logits_local [T, V_local] fp32 device, the global columns
 * [vocab_start, vocab_start + V_local); target [T] global; partials [3][T]
 * fp32 device output as above.  Merge with ce_merge_partials(S = T, B = 1);
 * rows_mean_f32 of the merged losses is ce_fwd_f32's mean.  One launch (the
 * flat CE row decompositions). */
int ce_partials_f32(const float* logits_local, const int64_t* target, int64_t T, int64_t V_local,
                    int64_t vocab_start, float* partials, void* stream);

/* ------------------------------------------------------------------------
 * Cross-entropy forward + backward: the losses and their gradient with
 * respect to the logits in one pass over HBM (logits read once, gradient
 * written once).  Same operations as ce_fwd_f32 / ce_fwd_sbv_bf16 (pages
 * "Cross-entropy loss" and "Vocab-parallel cross-entropy, Megatron layout",
 * section Semantics); the pages do not say whether their timings include the
 * backward, which is what training needs:
 *   dlogits[i, v] = g_i * (softmax(z_i)_v - [v == t_i]).
 * No mutation or aliasing: dlogits is a separate buffer the size of logits.
 * A target outside [0, V) makes that token's loss and gradient row NaN.
 *
 * ce_fwd_bwd_f32: flat fp32 [T, V]; g_i = grad_scale / T, i.e. dlogits is the
 *   gradient of grad_scale * loss with loss the mean.  loss [1] and the
 *   per-token losses in ws exactly as ce_fwd_f32 (ws >= ce_workspace_bytes,
 *   zeroed before first use).  dlogits fp32 [T, V] device output.
 * ce_fwd_bwd_sbv_bf16: Megatron layout bf16 [S, B, V]; per-token upstream
 *   gradients dloss fp32 [S, B] (device, or NULL for all ones) and
 *   g = grad_scale * dloss[s, b]; loss fp32 [S, B] as ce_fwd_sbv_bf16; dlogits
 *   bf16 [S, B, V] (round to nearest even).  No workspace.
 * grad_scale must be finite.  One kernel launch each.
 * ------------------------------------------------------------------------ */
int ce_fwd_bwd_f32(const float* logits, const int64_t* target, int64_t T, int64_t V,
                   float grad_scale, float* loss, float* dlogits, void* ws, size_t ws_bytes,
                   void* stream);
int ce_fwd_bwd_sbv_bf16(const uint16_t* logits, const int64_t* target, int64_t S, int64_t B,
                        int64_t V, const float* dloss, float grad_scale, float* loss,
                        uint16_t* dlogits, void* stream);

/* ------------------------------------------------------------------------
 * Fused linear + cross-entropy (logits z = x W^T never written to memory).
 * Page "Fused linear + CPO loss", summary ("computed chunked without
 * materializing logits") and section Semantics: x [batch, seq, hidden],
 * weight [vocab, hidden], target int64 [batch, seq], loss float [1]; bf16 per
 * its workload table.  Only the cross-entropy core is computed: the page does
 * not define the preference term.  Pass x flattened to [T = batch*seq, H].
 *
 *   x       [T, H] bf16 device, 16-byte aligned, H % 8 == 0
 *   W       [V, H] bf16 device, 16-byte aligned
 *   target  [T] int64 device
 *   loss    [1] fp32 device output: (1/T) sum_i loss_i; logits are accumulated
 *           in fp32 on the tensor cores and never rounded to bf16.
 *   ws      ws_bytes >= flce_workspace_bytes(T, H, V), zeroed before first
 *           use.  After completion the first T floats hold the per-token losses.
 * Status: LMHO_ERR_TIMEOUT is reported through lmho_ws_status().
 * ------------------------------------------------------------------------ */
size_t flce_workspace_bytes(int64_t T, int64_t H, int64_t V);
int flce_fwd_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t T,
                  int64_t H, int64_t V, float* loss, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Fused linear + cross-entropy, forward and backward.  Same loss as
 * flce_fwd_bf16 ("Fused linear + CPO loss", its cross-entropy core); the
 * gradients training needs, of grad_scale * loss (loss = the mean):
 *   dZ = (grad_scale / T) (softmax(x W^T) - onehot(target))   [T, V]
 *   dx = dZ W  [T, H] fp32 device output,  dW = dZ^T x  [V, H] fp32 device output
 * dZ is recomputed on the tensor cores from a second pass over the logit
 * tiles (after the forward pass gives each row's log-sum-exp), rounded to
 * bf16 (as the GEMM operand of the two gradient products) and kept in the
 * workspace; both products read it, W and x in place (no transposed copies);
 * the logits themselves are never stored.  When dx has too few output tiles
 * to fill the GPU (small T) its K range is split into fp32 slices summed in a
 * fixed order, so results stay bitwise reproducible.
 * x, W, dx, dW 16-byte aligned; H % 8 == 0.  grad_scale finite.  A target
 * outside [0, V) makes that token's loss, its dx row and all of dW NaN.
 *   ws   ws_bytes >= flce_bwd_workspace_bytes(T, H, V) (about 2 T V bytes beyond
 *        the forward's, plus up to 32 T H for the split slices when T H is
 *        small), zeroed before first use; the first T floats hold the per-token
 *        losses afterwards.
 * ------------------------------------------------------------------------ */
size_t flce_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V);
int flce_fwd_bwd_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t T,
                      int64_t H, int64_t V, float grad_scale, float* loss, float* dx, float* dW,
                      void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Fused linear + CPO loss: the whole objective of page "Fused linear + CPO
 * loss" (summary: CPO preference loss over batch x seq x hidden activations
 * projected through a vocab x hidden LM head against integer targets, logits
 * never materialised; Semantics: x [batch, seq, hidden], weight [vocab, hidden],
 * target int64 [batch, seq], loss float [1]).  The page does not print the
 * objective; this is the published CPO (Xu et al. 2024):
 *   sequence b < B/2 is the chosen answer of pair b, b + B/2 its rejected one;
 *   lp_b = sum_s ln softmax(x_{b,s} W^T)[t_{b,s}]   (all S tokens)
 *   loss = alpha * (token mean of the CE over the chosen half)
 *          + (2/B) sum_k -ln sigmoid(beta (lp_k - lp_{k+B/2})).
 *   x       [B, S, H] bf16 device (B even, >= 2), W [V, H] bf16 device
 *           (16-byte aligned, H % 8 == 0); target [B, S] int64 device
 *   beta    > 0 (0.1 in the paper), alpha >= 0 (1 in the paper), finite
 *   loss    [1] fp32 device output; logps [B] fp32 device output of lp, or NULL
 *   ws      ws_bytes >= flce_cpo_workspace_bytes(B, S, H, V), zeroed before
 *           first use; the first B*S floats hold the per-token CE losses.
 * A target outside [0, V) makes its token's loss, its sequence's lp and the
 * loss NaN.  One tensor-core pass (the fused CE) and two small finalisers.
 * ------------------------------------------------------------------------ */
size_t flce_cpo_workspace_bytes(int64_t B, int64_t S, int64_t H, int64_t V);
int flce_cpo_fwd_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t B,
                      int64_t S, int64_t H, int64_t V, float beta, float alpha, float* loss,
                      float* logps, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * flce_cpo_fwd_bf16 and the gradients of grad_scale * loss:
 *   dZ_i = grad_scale w_i (softmax(z_i) - onehot(t_i)),  w_i = d loss / d l_i
 *        = alpha/(Bc S) + (beta/Bc) sigmoid(-beta d_k)  (chosen token, pair k)
 *        = -(beta/Bc) sigmoid(-beta d_k)                (rejected token)
 *   with Bc = B/2, d_k = lp_k - lp_{k+Bc};  dx = dZ W [B*S, H] fp32,
 *   dW = dZ^T x [V, H] fp32 (as flce_fwd_bwd_bf16, dZ rounded to bf16).
 * dx, dW 16-byte aligned; ws_bytes >= flce_cpo_bwd_workspace_bytes(B, S, H, V),
 * zeroed before first use.  A bad target makes its pair's dx rows and all of
 * dW NaN.
 * ------------------------------------------------------------------------ */
size_t flce_cpo_bwd_workspace_bytes(int64_t B, int64_t S, int64_t H, int64_t V);
int flce_cpo_fwd_bwd_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t B,
                          int64_t S, int64_t H, int64_t V, float beta, float alpha, float grad_scale,
                          float* loss, float* logps, float* dx, float* dW, void* ws,
                          size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Fused linear + generalized Jensen-Shannon divergence, batchmean.
 * Page "Fused linear + JSD", summary (separate vocab x hidden heads for student
 * and teacher, generalized JSD with beta 0.5, batchmean) and section
 * Semantics: student_input [tokens, hidden], student_weight [vocab, hidden],
 * teacher_input, teacher_weight, loss float [1].
 *
 *   P = softmax(xs Ws^T) (student), Q = softmax(xt Wt^T) (teacher), per token;
 *   loss = (1/T) sum_i JSD_beta(P_i || Q_i).
 *
 *   xs, xt  [T, H] bf16 device;  Ws, Wt  [V, H] bf16 device (16-byte aligned,
 *           H % 8 == 0)
 *   beta    in (0, 1)
 *   loss    [1] fp32 device output
 *   ws      ws_bytes >= fljsd_workspace_bytes(T, H, V), zeroed before first
 *           use.  After completion the first T floats hold the per-token JSD.
 * Two tensor-core passes (log-sum-exp of both heads, then a recompute pass
 * that accumulates the divergence), since M couples both normalisers.
 * ------------------------------------------------------------------------ */
size_t fljsd_workspace_bytes(int64_t T, int64_t H, int64_t V);
int fljsd_fwd_bf16(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt,
                   const uint16_t* Wt, int64_t T, int64_t H, int64_t V, float beta,
                   float* loss, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * fljsd_fwd_bf16 with a temperature and a token mask (distillation variants;
 * the page names only beta 0.5 and batchmean, so these options are this
 * library's readings, and temperature 1 with no mask equals fljsd_fwd_bf16):
 *   P = softmax(xs Ws^T / temperature), Q = softmax(xt Wt^T / temperature);
 *   keep    [T] uint8 device, or NULL for all tokens: tokens with keep == 0
 *           contribute 0 and the batchmean divides by the number of kept
 *           tokens (a batch with no kept token has loss 0);
 *   temperature > 0 (finite reciprocal).  Other arguments as fljsd_fwd_bf16;
 *   the first T floats of ws hold the per-token JSD (0 for left-out tokens).
 * ------------------------------------------------------------------------ */
int fljsd_fwd_bf16_ex(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt,
                      const uint16_t* Wt, int64_t T, int64_t H, int64_t V, float beta,
                      float temperature, const uint8_t* keep, float* loss, void* ws,
                      size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Vocab-parallel fused losses: the vocabulary split of the page "Vocab-
 * parallel cross-entropy, Megatron layout" (summary: each tensor-parallel
 * rank holds its own vocab range) applied to the output layer.  A rank holds
 * the rows [vocab_start, vocab_start + V_local) of W (W_local [V_local, H]
 * bf16 device, 16-byte aligned), so its logits are x W_local^T; the full
 * inputs x / xs / xt [T, H] are on every rank.  Ranks exchange small per-token
 * results (all-gathers done by the caller, e.g. NCCL, in rank order); the
 * logits never leave the tensor cores.
 *
 * Fused linear + CE (pages "Fused linear + CPO loss", its cross-entropy core):
 * flce_partials_bf16: one shard.
 *   target    [T] int64 device, GLOBAL vocab indices
 *   partials  [3][T] fp32 device output, as ce_partials_sbv_bf16 writes them
 *             (m, s over the shard's logits; z = target logit or -inf)
 *   ws        ws_bytes >= flce_workspace_bytes(T, H, V_local), zeroed before
 *             first use.  Two launches (tensor-core pass, finaliser).
 * Then: all-gather the partials into [shards][3][T]; ce_merge_partials(...,
 * S = T, B = 1, V = global vocab, ...) gives the per-token losses, and
 * rows_mean_f32 their mean (the loss of flce_fwd_bf16 over the whole W, up to
 * rounding).
 *
 * Fused linear + generalized JSD (page "Fused linear + JSD"); beta,
 * temperature and the keep mask as fljsd_fwd_bf16_ex.  The divergence couples
 * both heads' normalisers, so there are two exchanges:
 * fljsd_lse_partials_bf16: shard pass 1.  lse_local [2][T] fp32 device
 *   output: each head's log-sum-exp of logits / temperature over the shard's
 *   columns (row 0 = student xs Ws_local^T, row 1 = teacher xt Wt_local^T).
 *   ws_bytes >= fljsd_workspace_bytes(T, H, V_local).  Two launches.
 * lse_merge_partials: [shards][2][T] fp32 device (the all-gather of the
 *   lse_local blocks, in rank order) -> lse [2][T] fp32 device, the global
 *   log-sum-exps: L = max_j l_j, lse = L + ln(sum_j exp(l_j - L)), in shard
 *   order.  One launch, no workspace.
 * fljsd_terms_bf16: shard pass 2.  lse [2][T] fp32 device = the global
 *   log-sum-exps; terms [T] fp32 device output: each token's sum over the
 *   shard's columns of beta P ln(P/M) + (1 - beta) Q ln(Q/M), with P, Q from
 *   the global normalisers.  kl_local [T] fp32 device, or NULL: with it, also
 *   each token's share of KL(P || M) over the shard's columns (needed by the
 *   backward below; the terms are the same bits either way).  ws as pass 1
 *   (the same workspace may serve both, one after the other).  Two launches.
 * jsd_merge_terms: [shards][T] fp32 device (the all-gather of the terms) ->
 *   rows [T] fp32 device (16-byte aligned): each token's JSD, the shards'
 *   sums added in shard order (0 where keep[i] == 0; keep [T] uint8 device or
 *   NULL); loss [1] fp32 device: their batchmean over the kept tokens (0 when
 *   none is kept).  Two launches, no workspace.
 * The shards must cover [0, V) exactly once (not checked); every shard uses
 * the same beta, temperature and inputs x.  Accumulation in fp32.
 * ------------------------------------------------------------------------ */
int flce_partials_bf16(const uint16_t* x, const uint16_t* W_local, const int64_t* target, int64_t T,
                       int64_t H, int64_t V_local, int64_t vocab_start, float* partials, void* ws,
                       size_t ws_bytes, void* stream);

/* flce_shard_bwd_bf16: the backward of one shard of the vocab-parallel fused
 * CE, gradients of grad_scale * (mean loss over the T tokens):
 *   dZ_shard = (grad_scale / T)(softmax(x W^T) - onehot(target)) restricted to
 *     the shard's columns, the softmax with each token's GLOBAL normaliser,
 *     taken from the gathered partials of the forward;
 *   dx_partial [T, H] fp32 = dZ_shard W_local: this rank's share of dx; the
 *     ranks' shares sum to dx (an all-reduce done by the caller);
 *   dW_local [V_local, H] fp32 = dZ_shard^T x: this rank's rows of dW.
 *   partials  [shards][3][T] fp32 device: every shard's flce_partials_bf16
 *             output in shard order (the forward's all-gather);
 *   V         the global vocabulary size (vocab_start + V_local <= V, else
 *             LMHO_ERR_INVALID_ARG): a target outside [0, V) makes that
 *             token's dZ row, and so dx's row and every dW entry, NaN;
 *   dx_partial, dW_local 16-byte aligned; ws_bytes >=
 *   flce_bwd_workspace_bytes(T, H, V_local), zeroed before first use.
 * dZ is rounded to bf16 for the two tensor-core products, as in
 * flce_fwd_bwd_bf16.  Launches: the normaliser merge, the dZ pass, the two
 * products (each with a K-slice sum when it splits K). */
int flce_shard_bwd_bf16(const uint16_t* x, const uint16_t* W_local, const int64_t* target,
                        const float* partials, int64_t shards, int64_t T, int64_t H, int64_t V_local,
                        int64_t vocab_start, int64_t V, float grad_scale, float* dx_partial,
                        float* dW_local, void* ws, size_t ws_bytes, void* stream);

/* flce_shard_bwd_rows_bf16: flce_shard_bwd_bf16 with a weight per token in
 * place of the mean's 1/T: dZ_shard row i = grad_scale * row_w[i] *
 * (softmax - onehot) over the shard's columns.  row_w [T] fp32 device (not
 * NULL), e.g. the CPO weights below.  Other arguments, workspace and launches
 * as flce_shard_bwd_bf16.
 *
 * cpo_combine_rows: the CPO objective (page "Fused linear + CPO loss"; the
 * published Contrastive Preference Optimization form, as flce_cpo_fwd_bf16)
 * of given per-token CE losses, e.g. the merged losses of the vocab-parallel
 * fused CE: rows [B * S] fp32 device, sequence b < B/2 chosen, b + B/2 its
 * rejected answer (B even >= 2); beta > 0, alpha >= 0 finite.
 *   loss  [1] fp32 device: alpha * (chosen NLL token mean) + mean softplus(-beta d_k);
 *   logps [B] fp32 device or NULL: each sequence's log-likelihood -sum_s rows;
 *   row_w [B * S] fp32 device or NULL: d loss / d rows_i, the weights of
 *         flce_shard_bwd_rows_bf16 for the CPO backward;
 *   ws    ws_bytes >= cpo_combine_workspace_bytes(B), 256-byte aligned, zeroed
 *         before first use.  One launch (a block per sequence, the last to
 *         finish combines the pairs in order). */
int flce_shard_bwd_rows_bf16(const uint16_t* x, const uint16_t* W_local, const int64_t* target,
                             const float* partials, int64_t shards, int64_t T, int64_t H,
                             int64_t V_local, int64_t vocab_start, int64_t V, const float* row_w,
                             float grad_scale, float* dx_partial, float* dW_local, void* ws,
                             size_t ws_bytes, void* stream);
size_t cpo_combine_workspace_bytes(int64_t B);
int cpo_combine_rows(const float* rows, int64_t B, int64_t S, float beta, float alpha, float* loss,
                     float* logps, float* row_w, void* ws, size_t ws_bytes, void* stream);
int fljsd_lse_partials_bf16(const uint16_t* xs, const uint16_t* Ws_local, const uint16_t* xt,
                            const uint16_t* Wt_local, int64_t T, int64_t H, int64_t V_local,
                            float temperature, float* lse_local, void* ws, size_t ws_bytes,
                            void* stream);
int lse_merge_partials(const float* parts, int64_t shards, int64_t T, float* lse, void* stream);
int fljsd_terms_bf16(const uint16_t* xs, const uint16_t* Ws_local, const uint16_t* xt,
                     const uint16_t* Wt_local, const float* lse, int64_t T, int64_t H,
                     int64_t V_local, float beta, float temperature, float* terms, float* kl_local,
                     void* ws, size_t ws_bytes, void* stream);
int jsd_merge_terms(const float* terms, int64_t shards, int64_t T, const uint8_t* keep,
                    float* rows, float* loss, void* stream);

/* fljsd_shard_bwd_bf16: the student's backward of one shard of the
 * vocab-parallel fused JSD, gradients of grad_scale * loss:
 *   lse [2][T] fp32 device   the global log-sum-exps (lse_merge_partials);
 *   kl  [T] fp32 device      each token's KL(P || M): the shards' kl_local
 *                            (fljsd_terms_bf16) all-gathered and summed, e.g.
 *                            by jsd_merge_terms without a mask (its rows);
 *   keep, beta, temperature  as for the forward;
 *   dxs_partial [T, H] fp32  this rank's share of the student's dx (the ranks'
 *                            shares sum to it: an all-reduce by the caller);
 *   dWs_local [V_local, H]   fp32, this rank's rows of the student's dW;
 *   dZs = (grad_scale / (n_kept temperature)) beta P (ln P - ln M - KL(P || M))
 *   over the shard's columns, rounded to bf16 for the two tensor-core products
 *   as in fljsd_fwd_bwd_bf16; left-out tokens contribute nothing.
 *   dxs_partial, dWs_local 16-byte aligned; ws_bytes >=
 *   fljsd_bwd_workspace_bytes(T, H, V_local), zeroed before first use.
 * Launches: the kept-token count and the dZ pass, the two products (each with
 * a K-slice sum when it splits K). */
int fljsd_shard_bwd_bf16(const uint16_t* xs, const uint16_t* Ws_local, const uint16_t* xt,
                         const uint16_t* Wt_local, const float* lse, const float* kl,
                         const uint8_t* keep, int64_t T, int64_t H, int64_t V_local, float beta,
                         float temperature, float grad_scale, float* dxs_partial, float* dWs_local,
                         void* ws, size_t ws_bytes, void* stream);

/* Deterministic mean of n fp32 values (rows 16-byte aligned, device) over
 * those with keep[i] != 0 (keep [n] uint8 device, or NULL = all; 0 when none
 * is kept) -> mean [1] fp32 device: compensated fp32 in a fixed order,
 * bitwise reproducible.  One launch, no workspace. */
int rows_mean_f32(const float* rows, int64_t n, const uint8_t* keep, float* mean, void* stream);

/* ------------------------------------------------------------------------
 * Fused linear + generalized JSD, forward and the student's backward (the
 * teacher is held fixed, as in distillation).  Loss as fljsd_fwd_bf16_ex;
 * gradients of grad_scale * loss with respect to the student input and head:
 *   dzs = (grad_scale / (n_kept temperature)) beta P (ln P - ln M - KL(P || M)),
 *   dxs = dZs Ws  [T, H] fp32,  dWs = dZs^T xs  [V, H] fp32,
 * (dJSD/dP = beta ln(P / M) through the softmax); left-out tokens contribute
 * nothing.  dZs is formed on the tensor cores from a third pass over both
 * heads' logit tiles, rounded to bf16 and kept in the workspace; the gradient
 * products read it as flce_fwd_bwd_bf16 does.  Arguments as
 * fljsd_fwd_bf16_ex; dxs, dWs 16-byte aligned;
 * ws_bytes >= fljsd_bwd_workspace_bytes(T, H, V), zeroed before first use.
 * ------------------------------------------------------------------------ */
size_t fljsd_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V);
int fljsd_fwd_bwd_bf16(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt,
                       const uint16_t* Wt, int64_t T, int64_t H, int64_t V, float beta,
                       float temperature, const uint8_t* keep, float grad_scale, float* loss,
                       float* dxs, float* dWs, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Device status of a workspace-carrying call (flce, fljsd).
 * Synchronises `stream`, reads the status word of `ws`, clears it, and returns
 * LMHO_OK or LMHO_ERR_TIMEOUT (a bounded wait inside a kernel gave up; that
 * call's outputs are then undefined).  ws_bytes must be the size passed to
 * the call.
 * ------------------------------------------------------------------------ */
int lmho_ws_status(void* ws, size_t ws_bytes, void* stream);

/* Row decomposition of the cross-entropy forward calls (ce_fwd_f32,
 * ce_fwd_f32_noalloc, ce_fwd_sbv_bf16, ce_partials_sbv_bf16), process-wide:
 *   0 = automatic (default): rows of at most 32 KB get a warp per row; longer
 *       rows a CTA per row, or a cluster of 8 CTAs per row when rows are few
 *       (< 4 per SM);
 *   1 = warp per row, 2 = CTA (256 threads) per row, 3 = CTA (512) per row,
 *   4 / 5 / 6 = cluster of 2 / 4 / 8 CTAs per row (DSMEM merge),
 *   7 = bulk-copy ring (rows up to 100 KB, 16-byte aligned; other rows fall
 *       back to a CTA per row).
 * Results agree to rounding whichever is chosen.  Returns LMHO_ERR_INVALID_ARG
 * for other values.  The environment variable LMHO_CE_VARIANT (warp, cta,
 * cta512, cluster2, cluster4, cluster8, bulk) sets the initial value. */
int lmho_set_ce_variant(int variant);

/* Raster of the fused-linear tensor-core passes, process-wide: work units
 * (token tile x vocab tile) are ordered in groups of `group_m` token tiles
 * of 128 (a paired pass's 256-row tiles count as two), vocab tiles outer
 * within a group, so the CTAs running at one time share W
 * tiles in L2; W streams from HBM about ceil(T/128/group_m) times per head
 * and pass.  0 = automatic: 32 for single-head passes, 16 for the two-head
 * JSD passes (both heads' tiles share L2) and for the gradient products;
 * otherwise 1..1024 for every pass.  Affects speed and DRAM traffic only,
 * never results.  Returns LMHO_ERR_INVALID_ARG outside that range. */
int lmho_set_raster_group(int group_m);

/* Measurement hook of the calling host thread: while set, every call that
 * thread makes records events[0] (a caller-created cudaEvent_t) on its stream
 * before its first kernel and events[i] after its i-th timed segment, for
 * i < n.  Segments per call: ce_fwd_f32 1 (the row kernel and its dependent
 * mean kernel together: an event between them would break their overlap),
 * ce_fwd_sbv_bf16 1, ce_partials_sbv_bf16 1, ce_merge_partials 1,
 * flce_fwd_bf16 2 (tensor-core pass, finaliser), fljsd_fwd_bf16 4
 * (log-sum-exp pass, finaliser, divergence pass, finaliser),
 * flce_partials_bf16, fljsd_lse_partials_bf16 and fljsd_terms_bf16 2 each
 * (tensor-core pass, finaliser), flce_shard_bwd_bf16 and
 * flce_shard_bwd_rows_bf16 3 (normaliser merge and dZ pass, dx share, dW
 * rows), cpo_combine_rows 1, fljsd_shard_bwd_bf16 3 (count and dZ pass, dxs
 * share, dWs rows), lse_merge_partials 1, jsd_merge_terms 1
 * (the merge and its dependent mean together), rows_mean_f32 1.  Calls made by
 * other threads are not affected.  Pass (NULL, 0) to turn it off. */
void lmho_set_launch_events(void* const* events, int n);

/* Bandwidth probe (a measurement aid; the operation pages have no such
 * operation): reads `segments` consecutive segments of segment_bytes (a
 * multiple of 16; data 16-byte aligned) with exactly the memory access of the
 * warp-per-row cross-entropy kernel (two-warp blocks, a warp per segment,
 * 16-byte streaming loads, 16 per lane in flight) and writes the XOR of each
 * segment's 32-bit words to out[segments] (uint32, device).  It computes
 * nothing else, so its time is the read-once floor that a cross-entropy call
 * over rows of that size can approach on this device.  One kernel launch. */
int lmho_probe_read(const void* data, int64_t segments, int64_t segment_bytes, uint32_t* out,
                    void* stream);

/* Host -> device copy by the SMs (a transfer utility of the library; no
 * operation page defines it).  Copies `bytes` from src, pinned (page-locked)
 * host memory with a device mapping (cudaHostAlloc, cudaMallocHost or
 * cudaHostRegister memory, as PyTorch's pin_memory gives), to dst, device
 * memory.  Both 16-byte aligned, bytes a multiple of 16, the two ranges
 * disjoint; bytes == 0 does nothing.  One kernel on `stream`, half the SMs x
 * 128 threads with 8 loads of 16 bytes in flight per thread; the copy engines
 * are not used, and no launch event is recorded.
 * Errors: LMHO_ERR_INVALID_ARG for a NULL pointer, a negative size or one not
 * a multiple of 16, misalignment, a src that is not pinned host memory, or a
 * dst that is not device (or managed) memory; LMHO_ERR_ALIAS if the ranges
 * overlap.
 * Why SM loads: on GB300 with a Grace host, copy-engine transfers from pinned
 * memory were slowed, in bursts lasting a few hundred milliseconds, while the
 * host served page faults caused by those transfers; SM loads fault only the
 * first time a buffer is read and then held the host link's rate.  At this
 * grid they run beside the library's tensor-core passes at ~205 GB/s. */
int lmho_copy_h2d(void* dst, const void* src, int64_t bytes, void* stream);

/* Upper bound, in nanoseconds, of every in-kernel wait of later calls
 * (default 2e9).  Process-wide. */
void lmho_set_wait_timeout_ns(uint64_t ns);

/* Self-test of the bounded-wait path: launches one block that waits on a
 * barrier nothing completes, for at most timeout_ns, then records
 * LMHO_ERR_TIMEOUT in the status word of ws (>= 256 bytes, zeroed).  Read it
 * back with lmho_ws_status(). */
int lmho_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* LMHO_H_ */
