/*
 * libeagle: the per-cycle dynamic draft-tree pipeline of EAGLE-2 speculative
 * decoding as hand-written CUDA kernels for sm_103a, behind a C ABI.
 *
 * Sources (page title and section):
 *   [summary]  "EAGLE-2: Faster Inference of Language Models with Dynamic
 *              Draft Trees" (paperlayer summary of arXiv 2406.16858v2),
 *              2.1 Speculative Sampling, 4.1 Expansion Phase, 4.2 Reranking
 *              Phase, App. A Implementation Details.
 *   [tutorial] "EAGLE-2: Dynamic Draft Trees" (stable-lab), "Value of a Node
 *              = Its Path Product", "Common misconception".
 *   [notes]    "EAGLE" (garden.houmin.site), EAGLE 方法 (TopK drafting, tree
 *              attention) and EAGLE 2 方法 (Expand with a threshold, ReRank
 *              with the shallower-node tie rule).
 *
 * One cycle, in call order:
 *   eagle_tree_init                       reset the tree state in `ws`
 *   eagle_lmhead (optional, per step)     LM-head logits of the frontier rows
 *   eagle_expand(step = 0 .. depth-1)     stages 1+2, one call per draft step
 *   eagle_rerank                          stage 3
 *   eagle_build_tree                      stage 4
 *   eagle_tree_attention                  stage 5 (one layer per call)
 *   eagle_verify                          stage 6
 *   eagle_kv_compact                      stage 6b
 *
 * Conventions for every call:
 *   - Pointers named in the signatures are device pointers owned by the
 *     caller unless stated; the library allocates nothing and keeps no state
 *     outside the caller's workspace, apart from cached device attributes.
 *   - Every call enqueues work on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns without synchronising; a whole cycle can be
 *     captured in a CUDA graph once each entry point has been called once
 *     outside capture (first calls set kernel attributes).
 *   - Argument checks run on the host before any launch; a failed check
 *     returns a negative eagle_status and launches nothing.
 *   - Faults found on the device (non-finite rows, out-of-range tokens or
 *     lengths, a bounded wait that gave up) set a status word in `ws`: the
 *     first error of the cycle wins, later kernels keep running, and outputs
 *     are undefined until eagle_status_fetch reports 0.
 *   - Rows of logits are contiguous; row starts must be 16-byte aligned
 *     (vocab * element size a multiple of 16, base pointer 16-byte aligned).
 *     A row holds at most 512 KB (vocab <= 262144 in bf16, 131072 in fp32):
 *     lossless verification keeps a whole row in the shared memory of one
 *     thread-block cluster.
 *   - Calls on distinct workspaces may run concurrently.
 */
#ifndef EAGLE_H_
#define EAGLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EAGLE_OK = 0,
    EAGLE_ERR_INVALID_ARG = -1, /* a host-side argument check failed */
    EAGLE_ERR_UNSUPPORTED = -2, /* valid but outside what the kernels support */
    EAGLE_ERR_LAUNCH = -3,      /* a CUDA launch or runtime call failed */
    EAGLE_ERR_WORKSPACE = -4,   /* workspace missing, misaligned or too small */
    EAGLE_ERR_DEVICE = -5,      /* eagle_status_fetch: the device raised an error */
    EAGLE_ERR_TIMEOUT = -6      /* eagle_status_fetch: a bounded device wait gave up */
} eagle_status;

typedef enum { EAGLE_F32 = 0, EAGLE_BF16 = 1 } eagle_dtype;

typedef enum { EAGLE_VERIFY_GREEDY = 0, EAGLE_VERIFY_LOSSLESS = 1, EAGLE_VERIFY_DRAFT = 2 } eagle_verify_mode;

/* Tree policy [summary 5.2.1, 5.2.2: the ablations of value-based expansion
 * and of reranking; tutorial "Watch the Budget Being Spent": the EAGLE-1
 * fixed shape against the dynamic tree]:
 *   EAGLE_POLICY_DYNAMIC     EAGLE-2: the frontier of each step is the top-k of
 *                            its children by path value; the rerank keeps the
 *                            N most valuable of all drafted nodes.
 *   EAGLE_POLICY_CONFIDENCE  the frontier is ranked by each child's own
 *                            confidence (its log-probability) instead of its
 *                            path value; the rerank is unchanged.
 *   EAGLE_POLICY_NO_RERANK   no rerank: the kept nodes are the ones the
 *                            expansion chose, the frontier of every step (k per
 *                            depth), the N most valuable of them if more.
 *   EAGLE_POLICY_STATIC      a fixed shape, the same for every input: the
 *                            frontier is chosen by position (child r of
 *                            frontier slot f ranked by f + r, then by lower
 *                            node id), and the kept nodes are the frontiers,
 *                            the first N by depth, then node id. */
typedef enum {
    EAGLE_POLICY_DYNAMIC = 0,
    EAGLE_POLICY_CONFIDENCE = 1,
    EAGLE_POLICY_NO_RERANK = 2,
    EAGLE_POLICY_STATIC = 3
} eagle_policy;

/* Draft-tree problem [summary 4.1, 4.2, App. A; notes EAGLE 2 方法]. */
typedef struct {
    int batch;       /* B, independent sequences */
    int vocab;       /* V, entries per logit row */
    int top_k;       /* k: children per expanded node and nodes expanded per step, 1..16 */
    int depth;       /* D: expansion steps = maximum draft depth, 1..16 */
    int node_budget; /* N: draft nodes kept by the rerank; tree slots T = N + 1 (root + N), T <= 256 */
    float threshold; /* path-value threshold below which a node is not expanded; <= 0 disables */
    int logit_dtype; /* eagle_dtype of the draft and target logits */
    int policy;      /* eagle_policy (0 = EAGLE-2) */
} eagle_tree_cfg;

/*
 * KV cache geometry (elements, not bytes). Element (b, layer, kv, pos, h, e)
 * with kv = 0 for K and 1 for V lives at
 *   b*seq_stride + layer*layer_stride + kv*kv_stride + pos*pos_stride + h*head_dim + e.
 * Tree slot j of sequence b is stored at position prefix_len[b] + j.
 */
typedef struct {
    int batch, n_q_heads, n_kv_heads, head_dim;
    int layers;  /* layers moved by eagle_kv_compact */
    int max_len; /* positions available per (sequence, layer, K|V) region */
    int dtype;   /* eagle_dtype of Q, K, V and the attention output */
    int64_t seq_stride, layer_stride, kv_stride, pos_stride;
} eagle_kv_cfg;

/* Candidate capacity C = k + (D-1) k^2 must be <= 1024. */

/* Bytes of the tree workspace for `cfg` (0 if cfg is invalid). The workspace
 * is device memory owned by the caller, 256-byte aligned, and must not be
 * shared by two cycles in flight. Its contents are opaque. */
size_t eagle_workspace_bytes(const eagle_tree_cfg* cfg);

/* Reset the per-cycle tree state: the root (depth 0) is the only frontier
 * node of step 0; no candidates. Clears nothing else. */
int eagle_tree_init(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, void* stream);

/*
 * Stages 1+2, draft step `step` (0-based) [notes EAGLE 方法: TopK drafting;
 * summary 4.1; tutorial "Value of a Node"; notes EAGLE 2 方法, Expand].
 *   draft_logits    [B, k, V] row f = the draft distribution of frontier slot f
 *                   of this step (step 0: only row 0, the root, is read; rows
 *                   f >= frontier count are never read).
 *   row_lse_in      [B, k] fp32 in, or NULL: the log-sum-exp of each row when
 *                   an upstream kernel already has it (e.g. an LM-head
 *                   epilogue); NULL = computed here (fp32, within 1e-5 of the
 *                   exact value at V = 128K).
 *   row_lse         [B, D, k] fp32 out: log-sum-exp used for each row read,
 *                   at [b, step, f]; NaN for rows not read.
 *   frontier_tokens [B, k] int32 out: tokens of the nodes to expand at step+1,
 *                   best value first, -1 padding (input of the next draft forward).
 *   frontier_count  [B] int32 out.
 * Per row: lse = max + log(sum exp(x - max)); the k largest logits (equal
 * logits: lower token id) become children with value
 * logv = logv(parent) + (x - lse) in fp32, logv(root) = 0. The next frontier
 * is the k highest-value children of this step among those with
 * logv >= log(threshold) (equal values: lower node id).
 */
int eagle_expand(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step, const void* draft_logits,
                 const float* row_lse_in, float* row_lse, int32_t* frontier_tokens, int32_t* frontier_count,
                 void* stream);

/*
 * Stages 1+2 with sampled drafting ["EAGLE-2: Faster Inference ..." summary,
 * 2.1 Speculative Sampling: the draft proposes tokens drawn from its
 * distribution]: the k children of frontier row f are drawn from the row's
 * softmax without replacement instead of being its k largest logits, by the
 * Gumbel-top-k identity: keys fl(x + g), g = -ln(-ln u) through a fixed-order
 * logarithm (atanh series, correctly rounded fp32 steps), u = ((word >> 9) +
 * 1/2) 2^-23; the children are the k largest keys in drawing order (equal
 * keys: lower id). The word of element x of row f of sequence b is word x % 4
 * of Philox4x32-10 at counter (x / 4, b * k + f, step, cycle & 0xffffffff)
 * under key (seed & 0xffffffff ^ 10, seed >> 32). Everything else (lse,
 * values from the unperturbed logits, threshold, frontier, outputs) is as
 * eagle_expand. With eagle_verify in EAGLE_VERIFY_DRAFT mode and a tree
 * shape that does not depend on the drawn tokens (EAGLE_POLICY_STATIC) the
 * cycle's output distribution is the target's.
 */
int eagle_expand_sampled(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step, const void* draft_logits,
                         const float* row_lse_in, uint64_t seed, uint64_t cycle, float* row_lse,
                         int32_t* frontier_tokens, int32_t* frontier_count, void* stream);

/*
 * LM head of a draft step, the projection whose rows stages 1+2 read
 * [notes EAGLE 方法: the draft model reuses the target model's LM head].
 *   hidden_dim      H, a multiple of 8 (>= 8).
 *   hidden          [B*k, H] bf16 in: row b*k + f is the draft model's last
 *                   hidden state for frontier slot f of sequence b (rows of
 *                   slots past the frontier count may hold anything finite).
 *   weight          [V, H] bf16 in: row v is vocabulary entry v's weights.
 *   draft_logits    [B, k, V] out, in cfg->logit_dtype: logits[r, v] =
 *                   sum_h hidden[r, h] * weight[v, h], accumulated in fp32
 *                   on the tensor cores (order and rounding of the fp32
 *                   sums unspecified; within H * 2^-23 * sum_h
 *                   |hidden[r, h] * weight[v, h]| of the exact sum), then
 *                   rounded to nearest even for bf16. The buffer
 *                   is the draft_logits argument of eagle_expand.
 * All three pointers 16-byte aligned; the weight stays read-only. Uses the
 * workspace's status word only (a timed-out wait raises it).
 */
int eagle_lmhead(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int hidden_dim, const void* hidden,
                 const void* weight, void* draft_logits, void* stream);

/*
 * LM head of a draft step with stage 1 in its epilogue [notes EAGLE 方法: the
 * draft model reuses the target's LM head, and TopK drafting reads its
 * distribution]: the logits of eagle_lmhead (fp32 tensor-core sums rounded to
 * cfg->logit_dtype) are reduced on chip and never written.
 *   hidden_dim, hidden, weight  as eagle_lmhead (B*k rows, bf16).
 *   scratch       device memory of eagle_lmhead_topk_scratch_bytes(cfg)
 *                 bytes, 256-byte aligned, owned by the caller: per-CTA
 *                 partials (max, sum of exp, top-k keys of each row);
 *                 contents undefined after the call.
 *   row_lse       [B*k] fp32 out: M + log(sum of exp(x - M)) over the row's
 *                 logits, fp32 (within 1e-5 of the exact value at V = 128K).
 *   topk_ids      [B*k, k] int32 out, topk_logits [B*k, k] fp32 out: the k
 *                 largest logits of each row as eagle_lmhead would store them
 *                 (equal logits: lower id), best first; -1 / -inf padding.
 * The outputs are those of eagle_shard_merge on the whole row and feed
 * eagle_expand_topk (topk_ids as [B, k, k], row_lse as [B, k]). Needs
 * B*k <= 4096 (EAGLE_ERR_UNSUPPORTED beyond). A non-finite lse raises
 * device status 1; a timed-out wait status 2.
 */
size_t eagle_lmhead_topk_scratch_bytes(const eagle_tree_cfg* cfg);
int eagle_lmhead_topk(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int hidden_dim, const void* hidden,
                      const void* weight, void* scratch, size_t scratch_bytes, float* row_lse, int32_t* topk_ids,
                      float* topk_logits, void* stream);

/*
 * Stage 3 [summary 4.2; tutorial "Value of a Node"; notes EAGLE 2 方法,
 * ReRank]: keep the min(N, #candidates) candidates with the largest value;
 * equal values keep the shallower node, then the lower node id. The kept set
 * is connected (every kept node's parent is kept or is the root). State stays
 * in `ws`.
 */
int eagle_rerank(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, void* stream);

/*
 * Stage 4 [summary 4.2: flattened sequence with a branch-separating mask].
 *   prefix_len [B] int32 in: verified tokens already in the KV cache (L_b).
 *   root_token [B] int32 in: last verified token (slot 0, depth 0).
 *   tokens, parent, depth, pos_ids [B, T] int32 out: slot 0 = root, slots
 *     1..n_tree-1 = kept nodes in node-id order (depth-major, so parents come
 *     first); parent = slot of the parent (-1 for the root); pos = L_b + depth;
 *     unused slots -1.
 *   mask [B, T, W] uint32 out, W = ceil(T/32): bit j of row i (word j/32,
 *     LSB first) is set iff slot j is an ancestor of slot i or i itself;
 *     unused rows are 0. The prefix is always visible and is not in the mask.
 *   n_tree [B] int32 out: 1 + kept nodes.
 */
int eagle_build_tree(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, const int32_t* prefix_len,
                     const int32_t* root_token, int32_t* tokens, int32_t* parent, int32_t* depth,
                     int32_t* pos_ids, uint32_t* mask, int32_t* n_tree, void* stream);

/*
 * Readout of the kept tree [tutorial, "Value of a Node = Its Path Product":
 * the expected number of accepted tokens of a verify pass is the sum of the
 * kept nodes' path values]. After eagle_rerank:
 *   value_sum [B] float out: sum over the kept nodes of exp(log path value),
 *   accumulated in fp32 in node-id order.
 */
int eagle_tree_value(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, float* value_sum, void* stream);

/* Scratch bytes for eagle_tree_attention with this geometry and T slots. */
size_t eagle_attention_workspace_bytes(const eagle_kv_cfg* kv, int T);

/*
 * Stage 5 [notes EAGLE 方法: tree attention verifies all branches at once;
 * summary 4.2]. For every sequence b, slot i < n_tree[b] and query head h:
 *   out[b,i,h,:] = sum_j softmax_j(q.k_j / sqrt(d)) v_j
 * over keys j in the prefix [0, L_b) and the tree slots set in mask row i
 * (cache position L_b + slot), KV head h / (Hq/Hkv). fp32 softmax and
 * accumulation; output in kv->dtype (bf16 rounds to nearest even). Rows
 * i >= n_tree[b] are written as zeros.
 *   q   [B, T, Hq, d] in, out [B, T, Hq, d] out, contiguous.
 *   kv_cache: base of the cache described by kv; `layer` selects the layer.
 *   ws/ws_bytes: attention scratch (eagle_attention_workspace_bytes), may
 *   alias nothing else in flight. Requires prefix_len[b] + T <= max_len.
 *   bf16 needs head_dim 128 (tensor-core path); fp32 supports head_dim <= 128.
 */
int eagle_tree_attention(const eagle_kv_cfg* kv, int T, const void* q, const void* kv_cache, int layer,
                         const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * Stage 6 [summary 2.1: target verification, tokens accepted sequentially by
 * the probability ratio; abstract: the output distribution is unchanged].
 *   seed, cycle     the uniforms of lossless verification are counter-based:
 *                   word c of sequence b (c = 0 .. T+1) is word 0 of
 *                   Philox4x32-10 (Salmon et al., SC'11) at counter
 *                   (c, b, cycle & 0xffffffff, cycle >> 32) under key
 *                   (seed & 0xffffffff ^ 7, seed >> 32), drawn on the device.
 *                   Word c tests the child at slot c (U24 = word >> 8); words T
 *                   and T+1 form U64 = w[T+1] * 2^32 + w[T] for the final
 *                   draw. Use a new cycle number per cycle. Unused by GREEDY.
 *   target_logits [B, T, V] in: the target's distribution at each slot.
 *   draft_logits  [D, B, k, V] in (DRAFT only, else may be NULL): the draft
 *                 rows of every step of the cycle, as passed to
 *                 eagle_expand_sampled; the workspace's frontiers map each
 *                 kept node to the row its children were drawn from.
 *   tokens, parent [B, T], n_tree [B] in: the tree from eagle_build_tree.
 *   accept_len [B] out: accepted draft tokens a_b (0..D).
 *   accepted_slots [B, D+1] out: slots of the accepted path, root first, -1 pad.
 *   out_tokens [B, D+1] out: the a_b accepted tokens then the bonus token, -1 pad.
 * GREEDY: the target's choice at slot t is argmax of row t (equal logits:
 *   lower id); walk from the root into the child carrying that choice.
 * LOSSLESS (temperature > 0): integer probabilities
 *   P_t[x] = floor(dexp((x - max_t) / temperature) * 2^40), dexp a fixed-order
 *   exp (Cody-Waite reduction, degree-7 Taylor in Horner form, each step one
 *   correctly rounded fp32 fused multiply-add); at node u the
 *   kept children are tested in slot order and child x is accepted iff
 *   U24 * S < 2^24 * P_u[x] (S = remaining mass); a rejection removes x. With
 *   no child accepted the bonus is the smallest token y (not removed) whose
 *   running mass exceeds floor(U64 * S / 2^64). Every row's maximum is taken
 *   in one pass over all rows; the masses of a row are summed only when the
 *   walk reaches its node (one cluster of CTAs per sequence).
 * DRAFT (temperature > 0; children drawn by eagle_expand_sampled): at node u
 *   with target residual A (initially P_u) and the remaining draft masses Q
 *   of u's draft row (integer masses as above, at the same temperature), the
 *   kept children are tested in slot (drawing) order and child x is accepted
 *   iff U24 * Q[x] * SA < 2^24 * A[x] * SQ (SA, SQ the sums); a rejection sets
 *   A[y] = floor(max(0, A[y] SQ - Q[y] SA) / 2^s) with s the smallest shift
 *   that brings the largest value to 2^40 or below (A is kept when all are 0),
 *   then removes x from Q. The bonus is the smallest y whose running sum of A
 *   exceeds floor(U64 * SA / 2^64). The walk runs in one cluster of CTAs per
 *   sequence; the residual is kept in the workspace.
 */
int eagle_verify(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int mode, float temperature, uint64_t seed,
                 uint64_t cycle, const void* target_logits, const void* draft_logits, const int32_t* tokens,
                 const int32_t* parent, const int32_t* n_tree, int32_t* accept_len, int32_t* accepted_slots,
                 int32_t* out_tokens, void* stream);

/*
 * Stage 6b: move the accepted path's KV into place (not on the pages: the
 * plain reading of compacting the accepted nodes' KV into the contiguous
 * cache after verification). For every layer in
 * [0, kv->layers), for K and V and j = 1..a_b:
 *   position L_b + j  <-  what position L_b + accepted_slots[b, j] held,
 * all sources read before any destination is written; positions outside
 * [L_b + 1, L_b + a_b] are untouched. new_len[b] = L_b + a_b + 1.
 *   accepted_slots [B, slots_stride] int32 (slots_stride >= max a_b + 1).
 *   ws: any eagle workspace whose status word receives device faults
 *   (a_b > 16, a slot s_j < j, or a position beyond max_len: that sequence
 *   is left untouched and new_len is not written); may be NULL.
 * Needs head_dim * n_kv_heads * element size and pos_stride * element size
 * to be multiples of 16 bytes.
 */
int eagle_kv_compact(const eagle_kv_cfg* kv, void* kv_cache, const int32_t* prefix_len, const int32_t* accept_len,
                     const int32_t* accepted_slots, int slots_stride, int32_t* new_len, void* ws, void* stream);

/* ------------------------------------------------- vocabulary shards --- */
/*
 * When the LM head is split over several GPUs by vocabulary rows, each GPU
 * holds a slice [vocab_offset, vocab_offset + shard_vocab) of every logit row
 * ["EAGLE" notes, EAGLE 方法: the top-k is taken over the whole vocabulary;
 * how the vocabulary is split is not on the pages]. Stage 1 and the greedy
 * verify then run on each slice into small partials, one exchange moves the
 * partials of all slices to every GPU (for example an all-gather: k keys and
 * two floats per row per slice), and eagle_shard_merge gives the whole row's
 * results; eagle_expand_topk and eagle_verify_argmax continue from them.
 *
 * A key is the 64-bit (order-preserving bits of the logit) << 32 |
 * (0xFFFFFFFF - token id): a larger key is a larger logit, then a lower token
 * id; 0 = no key.
 */

/* Stage-1 partials of `rows` logit rows of one slice.
 *   logits       [rows, shard_vocab] in cfg->logit_dtype, row starts 16-byte aligned.
 *   part_max_sum [rows, 2] fp32 out: the slice's maximum M_s and sum of exp(x - M_s).
 *   part_keys    [rows, 16] out: the slice's k largest keys, best first, 0 padding
 *                (token ids of the whole vocabulary: vocab_offset + index).
 * cfg->vocab is the whole vocabulary; vocab_offset + shard_vocab <= cfg->vocab. */
int eagle_shard_partials(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int rows, int shard_vocab,
                         int vocab_offset, const void* logits, float* part_max_sum, uint64_t* part_keys,
                         void* stream);

/* Merge of n_shards (<= 16) slices' partials, [n_shards, rows, ...] each:
 *   row_lse     [rows] fp32: M + log(sum_s S_s exp(M_s - M)), M = max_s M_s (the
 *               slices' terms added in slice order).
 *   topk_ids    [rows, k] int32, topk_logits [rows, k] fp32: the k largest logits
 *               of the whole row (equal logits: lower id), -1 / -inf padding.
 *   row_argmax  [rows] int32: the largest logit's token (lowest id on ties).
 * Equal to stage 1 of the whole row (top-k ids and argmax exactly; lse within
 * fp32 rounding of the unsplit row's). */
int eagle_shard_merge(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int n_shards, int rows,
                      const float* part_max_sum, const uint64_t* part_keys, float* row_lse, int32_t* topk_ids,
                      float* topk_logits, int32_t* row_argmax, void* stream);

/* Stage 2 of draft step `step` from merged stage-1 results (one CTA per
 * sequence): topk_ids / topk_logits [B, k, k] (row f = frontier slot f, as
 * eagle_shard_merge writes for the step's [B * k] rows), row_lse_in [B, k].
 * Children, values, threshold and next frontier exactly as eagle_expand. */
int eagle_expand_topk(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step, const int32_t* topk_ids,
                      const float* topk_logits, const float* row_lse_in, float* row_lse, int32_t* frontier_tokens,
                      int32_t* frontier_count, void* stream);

/* Greedy stage 6 from the target's argmax of every slot, row_argmax [B, T]
 * (merged over the slices): the walk and outputs of eagle_verify GREEDY. */
int eagle_verify_argmax(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, const int32_t* row_argmax,
                        const int32_t* tokens, const int32_t* parent, const int32_t* n_tree, int32_t* accept_len,
                        int32_t* accepted_slots, int32_t* out_tokens, void* stream);

/*
 * eagle_verify without a workspace, for callers that may not allocate device
 * memory (for example a plugin whose host engine plans all GPU memory up
 * front and forbids later allocations, or a decode loop that must never wait
 * on the allocator). No counterpart on the pages: it is the same stage 6 as
 * eagle_verify, with the same arguments and results, minus ws/ws_bytes.
 *   - Its per-row scratch is one fixed device array inside the library
 *     (about 70 KB, present on every GPU that loads the library until the
 *     process exits). It supports batch <= 1024 and batch * (node_budget + 1)
 *     <= 4096 rows in either mode and returns EAGLE_ERR_UNSUPPORTED beyond.
 *   - The first call on a device looks up that array's device address; make
 *     that first call before any stream capture. The address is kept per
 *     device for the life of the process: do not call this after
 *     cudaDeviceReset on that device.
 *   - Every call uses the same array, so calls that overlap on the GPU (on
 *     different streams, or from different threads) race and corrupt each
 *     other; serialise them. The array keeps the last call's contents; the
 *     call clears what must start at zero.
 *   - Device-detected faults are not reported (there is no workspace status
 *     word to read); bounds checks still keep every access in range.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
int eagle_verify_static(const eagle_tree_cfg* cfg, int mode, float temperature, uint64_t seed, uint64_t cycle,
                        const void* target_logits, const int32_t* tokens, const int32_t* parent,
                        const int32_t* n_tree, int32_t* accept_len, int32_t* accepted_slots, int32_t* out_tokens,
                        void* stream);

/* Synchronise `stream`, read the device status word of a workspace (the tree
 * workspace or the attention scratch: the word is the first 4 bytes of
 * either) into *device_status (0 = no fault, 1 non-finite row, 2 wait gave
 * up, 3 index out of range, 4 table overflow), clear it, and return EAGLE_OK,
 * EAGLE_ERR_DEVICE or EAGLE_ERR_TIMEOUT accordingly. */
int eagle_status_fetch(void* ws, int* device_status, void* stream);

/* ---------------------------------------------- inspection (tests, tools) --- */

/* Copy the candidate table and rerank result out of `ws` (device to device,
 * on `stream`): cand_* [B, C], kept [B, C] uint8, n_kept [B]. Any pointer may
 * be NULL. */
int eagle_tree_export(const eagle_tree_cfg* cfg, const void* ws, size_t ws_bytes, int32_t* cand_token,
                      int32_t* cand_parent, int32_t* cand_depth, float* cand_logv, uint8_t* cand_valid,
                      uint8_t* kept, int32_t* n_kept, void* stream);

/* Copy the per-row target statistics of the last eagle_verify: row maximum
 * [B, T] fp32, argmax [B, T] int32, integer mass sum_x P_t[x] [B, T] uint64
 * (lossless only: the rows of the nodes the walk visited, 0 for the others).
 * Rows t >= n_tree are unspecified. */
int eagle_verify_export(const eagle_tree_cfg* cfg, const void* ws, size_t ws_bytes, float* row_max,
                        int32_t* row_argmax, uint64_t* row_mass, void* stream);

/* Failure-path test hook: eagle_expand (own lse) with the row kernel's copy
 * producer switched off, so no copy is ever in flight and every consumer's
 * bounded wait on the chunk ring gives up (the first after about a second,
 * later ones at once). The launch completes, its outputs are meaningless and
 * the workspace's status word reads 2 (eagle_status_fetch returns
 * EAGLE_ERR_TIMEOUT); the context stays usable. */
int eagle_test_expand_starved(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step,
                              const void* draft_logits, float* row_lse, int32_t* frontier_tokens,
                              int32_t* frontier_count, void* stream);

/* The device arithmetic of sampled drafting, element by element: for i < n,
 * gumbel_out[i] = the Gumbel noise of words[i] and log_out[i] = the
 * fixed-order natural logarithm of ys[i] (positive normal floats), as
 * eagle_expand_sampled computes them. Either input may be NULL. */
int eagle_test_sampling(const uint32_t* words, const float* ys, int n, float* gumbel_out, float* log_out,
                        void* stream);

/* Kernels launched by this library since it was loaded (host-side count). */
uint64_t eagle_kernel_launches(void);

/* The cudaError_t of the calling thread's most recent call that returned
 * EAGLE_ERR_LAUNCH (0 if none), and its CUDA message in *message when
 * message is not NULL (a static string). */
int eagle_last_cuda_error(const char** message);

/* Human-readable message for an eagle_status value. */
const char* eagle_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE_H_ */
