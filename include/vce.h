/*
 * libvocabce — vocabulary-sharded embedding lookup and globally normalised
 * cross-entropy over a padded vocabulary, for one NVIDIA GB300 (sm_103a).
 *
 * C ABI. Every pointer argument except `p` is a DEVICE pointer owned by the
 * caller, unless a comment says otherwise. The library allocates no device
 * memory: scratch space is passed in as a caller-owned workspace whose size
 * `vce_workspace_size` returns. The library keeps no state between calls
 * apart from the wait limit set by `vce_set_wait_limit_ns` and a cache of
 * device attributes.
 *
 * All calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 * NULL is the legacy default stream). The return value reports argument,
 * shape, alignment and launch errors found on the host; nothing has been
 * enqueued when it is not VCE_OK. Data errors found on the device are
 * written to the optional `dev_status` word (int32, device memory, caller
 * sets it to 0): the first error wins (atomic compare-and-swap from 0).
 *
 * Sources are cited by page title and section:
 *  [VS]  "Vocabulary shards: look up locally and normalize globally",
 *        paragraphs 1-5.
 *  [PAD] "Training collapses when token embeddings are not padded to a
 *        multiple of 64", sections 4-7.
 *  [SPN] "Sequence-parallel normalization: shard tokens, retain their hidden
 *        features", paragraph 3.
 *  [TP]  "Tensor Parallelism (TP)", Component Sharding: Embedding
 *        (VocabDimShardedEmbedding) and LM Head (ColumnParallelLinear).
 */
#ifndef VCE_H
#define VCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vce_status {
  VCE_OK = 0,
  VCE_ERR_ARG = 1,          /* bad shape or argument (e.g. Vp not a multiple of 64) */
  VCE_ERR_UNSUPPORTED = 2,  /* valid but unsupported: dtype, alignment, size limit */
  VCE_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
  VCE_ERR_BAD_INDEX = 4,    /* device: a target outside [0,V_real) that is not ignore_index */
  VCE_ERR_TIMEOUT = 5,      /* device: a bounded wait inside a kernel ran out */
  VCE_ERR_WORKSPACE = 6     /* workspace missing, too small or misaligned */
} vce_status;

typedef enum vce_dtype {
  VCE_F32 = 0,   /* fp32 storage and fp32 arithmetic (SIMT FMA) */
  VCE_BF16 = 1   /* bf16 storage, fp32 accumulation on tcgen05 tensor cores */
} vce_dtype;

typedef enum vce_op {
  VCE_OP_EMBED_FWD = 0,
  VCE_OP_EMBED_BWD = 1,
  VCE_OP_LOSS_FWD = 2,
  VCE_OP_LOSS_BWD = 3,
  VCE_OP_SAMPLED_CANDIDATES = 4,
  VCE_OP_GREEDY_ARGMAX = 5
} vce_op;

/*
 * One problem. Shapes:
 *   h[T,H], W[Vp,H], E[T,H], dE[T,H]   row-major, element type `dtype`;
 *   ids[T], targets[T]                 int64;
 *   dW[Vp,H], dH[T,H]                  fp32, row-major (dH bf16 with
 *                                      VCE_FLAG_DH_BF16);
 *   lse[T], token_loss[T]              fp32;  owner maps int32.
 * Rows of every 2-D tensor are contiguous with stride H elements; H*size(dtype)
 * must be a multiple of 16 bytes and every 2-D tensor 16-byte aligned.
 *
 * Vocabulary layout [PAD s.5, s.7]: Vp is the padded vocabulary and must be a
 * multiple of 64; classes [0, V_real) are real, rows [V_real, Vp) are padding
 * and may hold any value (they are never read by the loss and never looked up).
 * Shards [TP, VS p.1]: S logical shards on one GPU; shard k owns the contiguous
 * rows [floor(k*Vp/S), floor((k+1)*Vp/S)). Any 1 <= S <= Vp is allowed.
 *
 * Limits: 0 <= T < 2^31, 1 <= H <= 65536, 64 <= Vp < 2^31, 1 <= V_real <= Vp,
 * and (T/256 + 1) * (Vp/256 + S) < 2^31 (the tensor-core kernels number their
 * work items in 32 bits); larger problems return VCE_ERR_UNSUPPORTED. The
 * embedding backward also needs T * ceil(H / (128 * 16 / sizeof(dtype))) < 2^31.
 * `flags` is 0 or a combination of the vce_flag bits below (other bits are
 * rejected with VCE_ERR_ARG).
 * ignore_index must lie outside [0, V_real): a value that names a real class
 * could not be told from a target of that class, so it is rejected with
 * VCE_ERR_ARG. The loss ignores targets equal to it, and an id equal to it is
 * the embedding's padding id (a zero row, no gradient).
 */
typedef struct vce_problem {
  int64_t T;
  int64_t H;
  int64_t Vp;
  int64_t V_real;
  int64_t ignore_index;   /* target value meaning "no loss here"; the usual -100 */
  int32_t S;
  int32_t tied_weights;   /* 1: embedding and LM head share W and one fp32 dW */
  int32_t dtype;          /* vce_dtype */
  int32_t flags;          /* vce_flag bits */
} vce_problem;

typedef enum vce_flag {
  /* vce_loss_bwd: add G W into dH instead of overwriting it. Lets a second
   * loss term on the same hidden states (the OT-H head of "Sampled Softmax with
   * Over-Tokenized Transformer", Setup: a second head on h[:-1] predicting
   * tokens[2:] at weight 0.1) accumulate its gradient into the first one's dH:
   * pass dH itself with T-1 rows and g = 0.1. */
  VCE_FLAG_ACCUMULATE_DH = 1,
  /* vce_loss_bwd, vce_sampled_loss: dH is bf16 [T,H] instead of fp32. The sum
   * over the vocabulary is kept in fp32 in the workspace and rounded to bf16
   * (nearest, ties to even) once; with VCE_FLAG_ACCUMULATE_DH the bf16 value
   * already in dH is added in fp32 before that rounding. */
  VCE_FLAG_DH_BF16 = 2
} vce_flag;

/* Bytes of workspace the call `op` needs for problem `p` (0 if none, SIZE_MAX
 * if the problem is invalid). The workspace must be 256-byte aligned. For
 * VCE_OP_LOSS_BWD this is the recommended size; any size of at least
 * vce_workspace_size_min(p, op) is accepted and a larger workspace lets the
 * backward process more vocabulary columns per pass. */
size_t vce_workspace_size(const vce_problem* p, int32_t op);
size_t vce_workspace_size_min(const vce_problem* p, int32_t op);

/*
 * Masked embedding lookup [VS p.1-2; TP Embedding, prefill].
 *   E[t,:] = W[ids[t],:]  if 0 <= ids[t] < V_real,   else 0.
 * The ownership test is done before any index into W is formed; the row is
 * owned by exactly one shard, so the sum over shards of the masked partial
 * lookups is the owner's row and the result is an exact copy.
 * Padding ids (ignore_index), negative ids, padded rows [V_real,Vp) and ids
 * >= Vp all give zero rows; they are not errors.
 * Optional outputs (NULL to skip): owner[t] = shard owning ids[t] (-1 if
 * invalid); local[t] = ids[t] - floor(owner*Vp/S) (-1 if invalid).
 * No workspace. `dev_status` is unused and may be NULL.
 */
vce_status vce_embed_fwd(const vce_problem* p, const int64_t* ids, const void* W,
                         void* E, int32_t* owner, int32_t* local,
                         int32_t* dev_status, void* stream);

/*
 * Embedding backward [VS p.2: repeated tokens accumulate into the same owned
 * row; tied weights combine all gradient contributions].
 *   dW[v,:] += sum over t with ids[t] == v of dE[t,:]      for 0 <= v < V_real
 * dW is fp32 and is always accumulated into (+=); rows with no valid id are
 * not touched. Invalid ids (as in vce_embed_fwd) contribute nothing.
 * Deterministic: valid (id, t) pairs are sorted ascending; the tokens of one
 * id are cut into runs of vce_embed_bwd_chunk() consecutive tokens; each run
 * is summed in fp32 from 0.0 in ascending t; the run sums are added left to
 * right; the total is added to dW[v] with one fp32 rounding. Results are
 * bit-identical run to run.
 * How the pairs are sorted does not change the result. Up to 16384 tokens the
 * ids are bucketed over the SMs. Above 8192 tokens, clusters of 8 CTAs share
 * the id loads through distributed shared memory (kernel kind
 * VCE_K_EMBED_SORT_CLUSTER); otherwise every CTA loads all ids itself
 * (VCE_K_EMBED_SORT). The environment variable VCE_EMBED_SORT_CLUSTER, read
 * at each call, overrides the choice: 1 for the clusters whenever the bucketed
 * counting sort runs, 0 for never.
 * Nor does the width of the column slices that the additions are cut into.
 * The runs of ids with more than one run are added in slices half as wide
 * when T * H * sizeof(dE element) is at most 64 MB (there the hottest id's
 * chain of dependent loads sets the call's time), else in the full width; the
 * environment variable VCE_EMBED_NARROW, read at each call, forces the half
 * width (1) or the full one (0). A plan records the width it was made for.
 * The call is vce_embed_bwd_plan followed by vce_embed_bwd_apply on the same
 * workspace, and it leaves the plan of `ids` there.
 * Workspace: vce_workspace_size(p, VCE_OP_EMBED_BWD) bytes.
 */
vce_status vce_embed_bwd(const vce_problem* p, const int64_t* ids, const void* dE,
                         float* dW, void* ws, size_t ws_bytes,
                         int32_t* dev_status, void* stream);

/*
 * The embedding backward in two parts [VS p.2: the tokens of one id
 * accumulate into its owned row]. The order of vce_embed_bwd depends on the
 * ids alone, so it can be worked out as soon as the ids are known (at the
 * lookup, for instance), before dE exists; only the application touches dE and
 * dW, which carry all of the backward's memory traffic.
 *
 * vce_embed_bwd_plan sorts the valid (id, t) pairs, cuts each id's tokens into
 * runs and writes this plan into `ws` (vce_workspace_size(p,
 * VCE_OP_EMBED_BWD) bytes), replacing whatever the workspace held. It reads
 * only `ids`. `dev_status` is unused and may be NULL.
 *
 * vce_embed_bwd_apply adds dE into dW by the plan held in `ws`, with exactly
 * the results of vce_embed_bwd for the planned ids (same order, same bits),
 * and leaves the plan unchanged: the same plan can be applied to another dE
 * or again. `p` must have the T, H and dtype the plan was made with; ids are
 * not passed again, and the caller must keep the plan's ids and workspace
 * together. A workspace that holds no plan, or one made for another T,
 * column count or V_real, adds nothing and reports VCE_ERR_ARG to dev_status
 * (the column count is that of the multi-run ids' slices: H, dtype and the
 * slice width enter through it, so a plan made under another
 * VCE_EMBED_NARROW setting can be refused). Two calls
 * on the same workspace must not overlap on the GPU (they share the plan's
 * counters).
 */
vce_status vce_embed_bwd_plan(const vce_problem* p, const int64_t* ids, void* ws,
                              size_t ws_bytes, int32_t* dev_status, void* stream);
vce_status vce_embed_bwd_apply(const vce_problem* p, const void* dE, float* dW,
                               void* ws, size_t ws_bytes, int32_t* dev_status,
                               void* stream);

/*
 * The lookup and the backward's plan in one call [VS p.1-2; TP Embedding]:
 * the results of vce_embed_fwd (E, owner, local) and of vce_embed_bwd_plan
 * (the plan in `ws`) for the same ids. The plan's sort reads only the ids and
 * moves almost no memory, so the lookup's row copies run beside it, on the
 * SMs the sort leaves free, instead of after it. The call completes, for any
 * later work on `stream`, only when both have. Arguments as in the two calls;
 * `dev_status` is unused and may be NULL.
 */
vce_status vce_embed_fwd_plan(const vce_problem* p, const int64_t* ids, const void* W,
                              void* E, int32_t* owner, int32_t* local, void* ws,
                              size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * Globally normalised cross-entropy, forward [VS p.3-5; PAD s.5; SPN p.3].
 *   z[t,v] = <h_t, W_v> accumulated in fp32, for real classes v < V_real only
 *   (padded classes are excluded, as if their logits were -inf);
 *   lse[t] = log sum_v exp(z[t,v]);  token_loss[t] = lse[t] - z[t, y_t];
 *   loss   = sum over valid t of token_loss[t] / N_valid   (0 if N_valid == 0).
 * A target y_t is valid iff 0 <= y_t < V_real. y_t == ignore_index is ignored.
 * Any other value is a data error: VCE_ERR_BAD_INDEX goes to dev_status and
 * the token is treated as ignored.
 * Each vocabulary tile's partial (max, sum of exp) and the target logit from
 * its unique owning tile are merged on the GPU into one maximum and one
 * denominator per token; the [T,Vp] logits are never written to memory.
 * Outputs: loss[1] and lse[T] (kept for the backward) are required;
 * token_loss[T] (0 for ignored tokens), target_owner[T] (shard owning y_t, -1
 * if not valid) and max_owner[T] (shard holding the largest logit, lowest shard
 * on ties) may be NULL. lse is written for every token.
 * Workspace: vce_workspace_size(p, VCE_OP_LOSS_FWD) bytes.
 */
vce_status vce_loss_fwd(const vce_problem* p, const void* h, const void* W,
                        const int64_t* targets, float* loss, float* lse,
                        float* token_loss, int32_t* target_owner, int32_t* max_owner,
                        void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * Cross-entropy backward [VS p.4: gradient = probability - target indicator,
 * times the loss scale; SPN p.3: averaged once over the valid tokens].
 *   G[t,v] = (exp(z[t,v] - lse[t]) - [v == y_t]) * g / N_valid
 * for valid t and real v, 0 elsewhere; z is recomputed tile by tile.
 *   dH  = G W        (fp32, or bf16 with VCE_FLAG_DH_BF16; overwritten, or
 *                     added into with VCE_FLAG_ACCUMULATE_DH)
 *   dW  = G^T h      rows [V_real,Vp) are 0:
 *         tied_weights == 0: dW is overwritten;
 *         tied_weights == 1: dW is accumulated into (+=), so that the embedding
 *         backward and this call combine into one parameter gradient.
 * lse must come from vce_loss_fwd on the same inputs. g is the upstream
 * gradient of the scalar loss (1 for a plain mean).
 * bf16: G is formed in bf16 for the two tensor-core GEMMs; fp32: all fp32.
 * Workspace: at least vce_workspace_size_min(p, VCE_OP_LOSS_BWD) bytes; the
 * vocabulary is processed in column chunks that fit the workspace. With
 * VCE_FLAG_DH_BF16 both sizes include T*H*4 bytes for the fp32 sum of dH.
 */
vce_status vce_loss_bwd(const vce_problem* p, const void* h, const void* W,
                        const int64_t* targets, const float* lse, float g,
                        void* dH, float* dW, void* ws, size_t ws_bytes,
                        int32_t* dev_status, void* stream);

/*
 * Candidate list of a sampled softmax ["Sampled Softmax with Over-Tokenized
 * Transformer", Setup: the loss scores the batch's targets plus random
 * negatives, P tokens in all, at each target's position in that list].
 *   cand[0 .. U)  the distinct valid targets (0 <= y < V_real), ascending;
 *   cand[U .. P)  the entries of `draws` that are not targets, in draw order;
 *   pos[t]        index of targets[t] in cand, or ignore_index when the target
 *                 is ignored or invalid;  *n_unique = U.
 * `draws` (device, n_draws int64) are the method's random numbers, uniform
 * over [0, V_real) (e.g. a prefix of a random permutation). Negatives are
 * drawn without replacement: a draw that is a target, repeats an earlier
 * negative or lies outside [0, V_real) is skipped, so cand holds distinct ids. Uses p->T, p->V_real
 * and p->ignore_index. cand[P], pos[T] int64 and n_unique (one int32) are
 * device outputs. Data errors go to dev_status: a target that is neither
 * valid nor ignore_index -> VCE_ERR_BAD_INDEX (treated as ignored); U > P or
 * too few usable draws -> VCE_ERR_ARG; the unfilled entries of cand are then
 * -1 (and, when U > P, every entry of cand is -1 and every pos ignore_index).
 * Workspace: vce_workspace_size(p, VCE_OP_SAMPLED_CANDIDATES) bytes.
 */
vce_status vce_sampled_candidates(const vce_problem* p, const int64_t* targets, const int64_t* draws,
                                  int64_t n_draws, int64_t P, int64_t* cand, int64_t* pos,
                                  int32_t* n_unique, void* ws, size_t ws_bytes, int32_t* dev_status,
                                  void* stream);

/*
 * Sampled-softmax loss, forward and backward in one call ["Sampled Softmax
 * with Over-Tokenized Transformer", Setup and its loss listing: the head's
 * logits are taken over W[cand] only and the cross-entropy is taken at
 * position_in(cand, target)]. In order, on `stream`:
 *   1. vce_sampled_candidates  -> cand[P], pos[T], *n_unique
 *   2. Wc = W[cand]            (vce_embed_fwd with T = P, ids = cand; a [P, H]
 *                               table in the workspace, padded to 64 rows)
 *   3. the globally normalised cross-entropy over the P candidate columns
 *      (vce_loss_fwd with Vp = P rounded up to 64, V_real = P, S = 1,
 *      targets = pos) -> *loss (mean over valid tokens), lse[T]
 *   4. its backward (vce_loss_bwd, untied) -> dH[T,H] overwritten (added
 *      into when p->flags has VCE_FLAG_ACCUMULATE_DH; bf16 with
 *      VCE_FLAG_DH_BF16), and the
 *      candidate rows' gradient dWc[P,H] in the workspace
 *   5. dW[cand[i], :] += dWc[i, :], one fp32 addition per element (the
 *      candidates are distinct); rows of dW that are not candidates, and
 *      entries of cand that are -1, are untouched.
 * p describes the full problem (T, H, Vp, V_real, S, dtype, ignore_index; its
 * tied_weights is ignored: dW is always accumulated into). h[T,H] and W[Vp,H]
 * in p->dtype, dW[Vp,H] fp32, g the upstream gradient of the mean loss.
 * lse may be NULL (kept in the workspace). Statuses and data errors as for the
 * five steps; dev_status collects the first data error of any of them.
 * Workspace: vce_sampled_workspace_size(p, P) bytes recommended; less is
 * accepted down to the size that lets the backward run in 256-column chunks.
 */
size_t vce_sampled_workspace_size(const vce_problem* p, int64_t P);
vce_status vce_sampled_loss(const vce_problem* p, const void* h, const void* W, const int64_t* targets,
                            const int64_t* draws, int64_t n_draws, int64_t P, float g, float* loss,
                            float* lse, void* dH, float* dW, int64_t* cand, int64_t* pos,
                            int32_t* n_unique, void* ws, size_t ws_bytes, int32_t* dev_status,
                            void* stream);

/*
 * Greedy decoding over the sharded head ["Tensor Parallelism (TP)", on-device
 * sampling: the sampler finds the global argmax across the TP-sharded logits
 * without gathering them; "Vocabulary shards ...", paragraph 3: maxima are
 * taken over valid entries only]. For every token t, with z = h W^T:
 *   argmax[t]    = the lowest v in [0, V_real) with z_tv = max_u z_tu (int64);
 *   max_logit[t] = that logit (fp32; optional);
 *   owner[t]     = the shard owning argmax[t] (int32; optional).
 * Padded classes [V_real, Vp) never win. Each shard's work units report their
 * (max, lowest column); the pairs are merged on the GPU. No targets, no loss.
 * Uses p->T, H, Vp, V_real, S and dtype. argmax must not be NULL when T > 0.
 * Workspace: vce_workspace_size(p, VCE_OP_GREEDY_ARGMAX) bytes.
 */
vce_status vce_greedy_argmax(const vce_problem* p, const void* h, const void* W, int64_t* argmax,
                             float* max_logit, int32_t* owner, void* ws, size_t ws_bytes,
                             int32_t* dev_status, void* stream);

/*
 * Hashed n-gram input embeddings ["Sampled Softmax with Over-Tokenized
 * Transformer", Setup and its loss listing: each input token's embedding gains
 * the hashed 2-gram and 3-gram embeddings that end at it].
 * The n-gram ending at token t of the input ids x is (x[t-n+1], ..., x[t]); its
 * row in a table of M rows is the n-gram read as a base-V number (x[t] the
 * lowest digit) mod M:
 *     idx_n(t) = (x[t] + x[t-1]*V + ... + x[t-n+1]*V^(n-1)) mod M,   V = V_real.
 * A token with fewer than n-1 earlier tokens in its sequence (the ids are
 * sequences of seq_len tokens laid end to end; seq_len = 0: one sequence), or
 * whose n-gram holds an id outside [0, V_real), has no n-gram: index -1.
 *
 * vce_ngram_hash: out[t] = idx_n(t) (int64, device) for n >= 1, 1 <= M < 2^31,
 * 1 <= V < 2^31.
 */
vce_status vce_ngram_hash(const int64_t* ids, int64_t T, int32_t n, int64_t V, int64_t M, int64_t seq_len,
                          int64_t* out, void* stream);

/*
 * E[t] = W[x_t] + T2[idx_2(t)] + T3[idx_3(t)], summed in fp32 in that order (a
 * missing term, an invalid id or an absent n-gram, reads as +0) and rounded
 * once to p->dtype (round to nearest even). W[Vp,H], T2[M2,H], T3[M3,H] and
 * E[T,H] in p->dtype, 16-byte aligned. M2 = 0 (T2 NULL) or M3 = 0 (T3 NULL)
 * leaves that table out. Uses p->T, H, V_real, dtype; ids are the input ids.
 */
vce_status vce_ngram_embed_fwd(const vce_problem* p, const int64_t* ids, const void* W, const void* T2,
                               int64_t M2, const void* T3, int64_t M3, int64_t seq_len, void* E,
                               int32_t* dev_status, void* stream);

/*
 * Backward of vce_ngram_embed_fwd: dW[x_t] += dE[t], dT2[idx_2(t)] += dE[t],
 * dT3[idx_3(t)] += dE[t] (fp32 tables, accumulated into), each with the
 * deterministic order of vce_embed_bwd (sorted (row, t), runs of 32 tokens
 * summed in fp32, run sums left to right, one rounding into the row), so the
 * results are bit-identical from run to run. dT2 / dT3 may be NULL when M2 /
 * M3 is 0. Workspace: vce_ngram_workspace_size(p) bytes.
 */
size_t vce_ngram_workspace_size(const vce_problem* p);
vce_status vce_ngram_embed_bwd(const vce_problem* p, const int64_t* ids, const void* dE, float* dW, float* dT2,
                               int64_t M2, float* dT3, int64_t M3, int64_t seq_len, void* ws, size_t ws_bytes,
                               int32_t* dev_status, void* stream);

/*
 * vce_ngram_embed_bwd in two parts ["Sampled Softmax with Over-Tokenized
 * Transformer", Setup; VS p.2], as vce_embed_bwd_plan / _apply are for the
 * token table: the plan (the tables' row indices and the sort of every
 * table's (row, t) pairs) depends on the ids alone; the application adds dE
 * into dW, dT2 and dT3 by it, with the bits of vce_ngram_embed_bwd, and leaves
 * the plan unchanged. vce_ngram_embed_bwd also leaves its plan in `ws`. The
 * application must pass the p, M2 and M3 of the plan; a table whose part of
 * the workspace holds no plan of this T, column count and row count adds
 * nothing to any table and reports VCE_ERR_ARG to dev_status. Workspace:
 * vce_ngram_workspace_size(p) bytes for both.
 */
vce_status vce_ngram_embed_bwd_plan(const vce_problem* p, const int64_t* ids, int64_t M2, int64_t M3,
                                    int64_t seq_len, void* ws, size_t ws_bytes, int32_t* dev_status,
                                    void* stream);
vce_status vce_ngram_embed_bwd_apply(const vce_problem* p, const void* dE, float* dW, float* dT2, int64_t M2,
                                     float* dT3, int64_t M3, void* ws, size_t ws_bytes, int32_t* dev_status,
                                     void* stream);

/*
 * Loss forward without a caller workspace. The method's pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory (a plugin inside a framework that owns all device memory and hands it
 * only inputs and outputs, or a hot path that must not call cudaMalloc).
 * Computes exactly what vce_loss_fwd computes, with the same kernels and the
 * same arguments minus the workspace. Its scratch is a fixed array of
 * vce_loss_fwd_noalloc_max_scratch() bytes (16 MiB) in the library's own
 * device memory, held on every GPU that loads the library until the process
 * exits; a problem whose forward workspace (vce_workspace_size(p,
 * VCE_OP_LOSS_FWD)) is larger returns VCE_ERR_WORKSPACE before anything is
 * enqueued. No device memory is allocated by the call.
 * It takes the same problems, flags and pointers as vce_loss_fwd and checks
 * them by the same rules; on a refusal for size, vce_last_error() names the
 * scratch the problem needs and the array's size.
 * The first call on a device looks up the array's device address for that
 * device (the device must be current) and keeps it; make that first call
 * before any stream capture. A device reset after it is not supported (the
 * kept address would be stale). All calls share the one array: calls that may
 * overlap on the GPU (different streams without ordering, or different host
 * threads) race on it and must not be used. When dev_status is NULL the status
 * word inside the array is cleared at the start of each call.
 */
vce_status vce_loss_fwd_noalloc(const vce_problem* p, const void* h, const void* W,
                                const int64_t* targets, float* loss, float* lse,
                                float* token_loss, int32_t* target_owner, int32_t* max_owner,
                                int32_t* dev_status, void* stream);
size_t vce_loss_fwd_noalloc_max_scratch(void);

/* Static string naming a status code. */
const char* vce_status_str(vce_status s);

/* Name and text of the CUDA error behind the calling thread's last
 * VCE_ERR_CUDA, or the reason for vce_loss_fwd_noalloc's last refusal for
 * size ("" if none); thread-local storage, valid until the thread's next
 * call. */
const char* vce_last_error(void);

/* The run length of the embedding backward's fixed summation order (tokens). */
int32_t vce_embed_bwd_chunk(void);

/* Library version, major*10000 + minor*100 + patch. */
int32_t vce_version(void);

/*
 * Upper bound, in nanoseconds, on any single wait inside a kernel (pipeline
 * barriers of the tensor-core kernels). When a wait runs out the kernel stops
 * its work, writes VCE_ERR_TIMEOUT to dev_status (or to the workspace's status
 * word when dev_status is NULL) and returns. Default 2e9 (2 s). Process-wide.
 */
void vce_set_wait_limit_ns(uint64_t ns);

/*
 * Self-test of the bounded wait: launches one block that waits on a pipeline
 * barrier nothing will ever complete, bounded by `limit_ns`. The kernel gives
 * up, writes VCE_ERR_TIMEOUT to dev_status and exits; the stream and context
 * stay usable. Used by the failure-detection tests. No workspace.
 */
vce_status vce_wait_selftest(uint64_t limit_ns, int32_t* dev_status, void* stream);

/*
 * Launch accounting, for profilers and benchmarks (no counterpart on the
 * pages). Every kernel the library launches increments a process-wide
 * counter (vce_launch_count).
 *
 * Per-launch timing: vce_profile_begin(capacity, stream) creates `capacity`
 * timing events (host-side CUDA event objects, no device memory) and records
 * a start event on `stream`. Until vce_profile_end, every kernel launch made by
 * the library records the next event on its own stream right after itself.
 * vce_profile_end waits for the last recorded event, writes for each launch i
 * its vce_kernel_kind and the milliseconds between event i-1 (the start event
 * for i = 0) and event i, destroys the events and returns the number of
 * launches recorded (at most `capacity`, -1 on error). Launches on one stream
 * run back to back, so each interval is that launch's duration including its
 * launch gap. Process-wide; not for concurrent callers.
 * VCE_K_LOSS_MEAN and VCE_K_DH_REDUCE keep their numbers but are no longer
 * launched (the merge's last block takes the mean; the dH K parts are added
 * inside the DH kernel); VCE_K_COUNT_VALID is launched by the fp32 path only.
 */
typedef enum vce_kernel_kind {
  VCE_K_EMBED_GATHER = 0, VCE_K_EMBED_SORT = 1, VCE_K_EMBED_REDUCE = 2,
  VCE_K_TC_FWD = 3, VCE_K_TC_GRAD = 4, VCE_K_TC_DH = 5, VCE_K_TC_DW = 6,
  VCE_K_MERGE = 7, VCE_K_LOSS_MEAN = 8, VCE_K_COUNT_VALID = 9,
  VCE_K_SIMT_FWD = 10, VCE_K_SIMT_GRAD = 11, VCE_K_SGEMM = 12, VCE_K_WAIT_SELFTEST = 13,
  VCE_K_DH_REDUCE = 14, VCE_K_SAMPLED_CAND = 15, VCE_K_SAMPLED_SCATTER = 16,
  VCE_K_TC_ARGMAX = 17, VCE_K_ARGMAX_MERGE = 18, VCE_K_SIMT_ARGMAX = 19,
  VCE_K_NGRAM_HASH = 20, VCE_K_NGRAM_FWD = 21, VCE_K_EMBED_HDR = 22, VCE_K_DH_BF16 = 23,
  VCE_K_EMBED_SORT_CLUSTER = 24
} vce_kernel_kind;
uint64_t vce_launch_count(void);
vce_status vce_profile_begin(int32_t capacity, void* stream);
int32_t vce_profile_end(float* ms, int32_t* kinds, int32_t capacity);

#ifdef __cplusplus
}
#endif

#endif /* VCE_H */
