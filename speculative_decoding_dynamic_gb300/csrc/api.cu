// C-ABI entry points of libeagle: argument checks, workspace layout, launches.
// Declarations and the contract of every call are in include/eagle.h.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "../../include/eagle.h"
#include "eagle_ws.h"

namespace eagle {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

cudaError_t launch_attention_simt(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                                  const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                                  int* status, cudaStream_t stream);

}  // namespace eagle

using namespace eagle;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Resolve and check a tree configuration. Returns EAGLE_OK or an error.
int resolve(const eagle_tree_cfg* cfg, TreeDims* d) {
    if (cfg == nullptr) return EAGLE_ERR_INVALID_ARG;
    const int B = cfg->batch, V = cfg->vocab, k = cfg->top_k, D = cfg->depth, N = cfg->node_budget;
    if (B < 1 || B > 65535 || k < 1 || k > kMaxTopK || D < 1 || D > kMaxDepth || N < 1) return EAGLE_ERR_INVALID_ARG;
    if (V < k) return EAGLE_ERR_INVALID_ARG;
    if (cfg->logit_dtype != EAGLE_F32 && cfg->logit_dtype != EAGLE_BF16) return EAGLE_ERR_INVALID_ARG;
    if (std::isnan(cfg->threshold)) return EAGLE_ERR_INVALID_ARG;
    if (cfg->policy < EAGLE_POLICY_DYNAMIC || cfg->policy > EAGLE_POLICY_STATIC) return EAGLE_ERR_INVALID_ARG;
    const long C = k + static_cast<long>(D - 1) * k * k;
    const int T = N + 1;
    if (C > kMaxCandidates || T > kMaxSlots) return EAGLE_ERR_UNSUPPORTED;
    const int esize = cfg->logit_dtype == EAGLE_BF16 ? 2 : 4;
    if ((static_cast<long>(V) * esize) % 16 != 0) return EAGLE_ERR_UNSUPPORTED;
    // lossless verification keeps a row resident over one cluster: V * esize <= 8 * 4 * 16 KB
    if (row_chunks(row_seg_elems(V, esize, kMaxChunks), esize) > kRowStages) return EAGLE_ERR_UNSUPPORTED;
    if (static_cast<long>(B) * (T > k ? T : k) > 65535) return EAGLE_ERR_UNSUPPORTED;  // grid.y
    d->B = B;
    d->V = V;
    d->k = k;
    d->D = D;
    d->N = N;
    d->T = T;
    d->W = (T + 31) / 32;
    d->C = static_cast<int>(C);
    d->log_thr = cfg->threshold > 0.0f ? static_cast<float>(std::log(static_cast<double>(cfg->threshold)))
                                       : -INFINITY;
    d->dtype = cfg->logit_dtype;
    d->policy = cfg->policy;
    return EAGLE_OK;
}

int bind_ws(const TreeDims& d, const void* ws, size_t ws_bytes, TreeWs* w) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return EAGLE_ERR_WORKSPACE;
    const size_t need = ws_layout(d, nullptr, nullptr);
    if (ws_bytes < need) return EAGLE_ERR_WORKSPACE;
    ws_layout(d, const_cast<void*>(ws), w);
    return EAGLE_OK;
}

int resolve_kv(const eagle_kv_cfg* kv, KvDims* k) {
    if (kv == nullptr) return EAGLE_ERR_INVALID_ARG;
    if (kv->batch < 1 || kv->n_q_heads < 1 || kv->n_kv_heads < 1 || kv->head_dim < 1 || kv->layers < 0 ||
        kv->max_len < 1)
        return EAGLE_ERR_INVALID_ARG;
    if (kv->n_q_heads % kv->n_kv_heads != 0) return EAGLE_ERR_INVALID_ARG;
    if (kv->dtype != EAGLE_F32 && kv->dtype != EAGLE_BF16) return EAGLE_ERR_INVALID_ARG;
    if (kv->seq_stride < 0 || kv->layer_stride < 0 || kv->kv_stride < 0 || kv->pos_stride < 1)
        return EAGLE_ERR_INVALID_ARG;
    if (kv->pos_stride < static_cast<int64_t>(kv->n_kv_heads) * kv->head_dim) return EAGLE_ERR_INVALID_ARG;
    k->B = kv->batch;
    k->Hq = kv->n_q_heads;
    k->Hkv = kv->n_kv_heads;
    k->d = kv->head_dim;
    k->layers = kv->layers;
    k->max_len = kv->max_len;
    k->dtype = kv->dtype;
    k->seq_stride = kv->seq_stride;
    k->layer_stride = kv->layer_stride;
    k->kv_stride = kv->kv_stride;
    k->pos_stride = kv->pos_stride;
    return EAGLE_OK;
}

// The CUDA error of the calling thread's last failed call (0 = none).
thread_local int g_last_cuda_error = 0;

// One C-ABI call: an NVTX range named after the call (for profilers; a null
// check when no tool is attached), and the stream and workspace that a
// checked build waits on.
thread_local cudaStream_t g_call_stream = nullptr;
thread_local const void* g_call_ws = nullptr;
struct CallScope {
    CallScope(const char* name, void* stream, const void* ws) {
        nvtxRangePushA(name);
        g_call_stream = static_cast<cudaStream_t>(stream);
        g_call_ws = ws;
    }
    ~CallScope() { nvtxRangePop(); }
};
#define EAGLE_CALL(stream, ws) CallScope eagle_call_scope_(__func__, (stream), (ws))

int launch_result(cudaError_t e) {
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        return EAGLE_ERR_LAUNCH;
    }
#ifdef EAGLE_DEBUG
    // Checked builds: the call waits for its work (outside stream capture) and
    // reports a fault of its own kernels: a failed execution, or the
    // workspace's status word (left set for eagle_status_fetch).
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(g_call_stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
        return EAGLE_OK;
    cudaError_t se = cudaStreamSynchronize(g_call_stream);
    if (se != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(se);
        return EAGLE_ERR_LAUNCH;
    }
    if (g_call_ws != nullptr) {
        int v = 0;
        if (cudaMemcpy(&v, g_call_ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return EAGLE_ERR_LAUNCH;
        if (v != 0) return v == 2 ? EAGLE_ERR_TIMEOUT : EAGLE_ERR_DEVICE;
    }
#endif
    return EAGLE_OK;
}

}  // namespace

extern "C" {

size_t eagle_workspace_bytes(const eagle_tree_cfg* cfg) {
    TreeDims d;
    if (resolve(cfg, &d) != EAGLE_OK) return 0;
    return ws_layout(d, nullptr, nullptr);
}

int eagle_tree_init(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    return launch_result(launch_tree_init(d, w, static_cast<cudaStream_t>(stream)));
}

static int expand_call(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step, const void* draft_logits,
                       const float* row_lse_in, float* row_lse, int32_t* frontier_tokens, int32_t* frontier_count,
                       void* stream, bool starve, const uint64_t* sample_seed_cycle = nullptr) {
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (step < 0 || step >= d.D) return EAGLE_ERR_INVALID_ARG;
    if (!draft_logits || !row_lse || !frontier_tokens || !frontier_count) return EAGLE_ERR_INVALID_ARG;
    if (!aligned16(draft_logits)) return EAGLE_ERR_UNSUPPORTED;
    return launch_result(launch_expand(d, w, step, draft_logits, row_lse_in, row_lse, frontier_tokens,
                                       frontier_count, static_cast<cudaStream_t>(stream), starve, sample_seed_cycle));
}

int eagle_expand(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step, const void* draft_logits,
                 const float* row_lse_in, float* row_lse, int32_t* frontier_tokens, int32_t* frontier_count,
                 void* stream) {
    EAGLE_CALL(stream, ws);
    return expand_call(cfg, ws, ws_bytes, step, draft_logits, row_lse_in, row_lse, frontier_tokens, frontier_count,
                       stream, false);
}

int eagle_expand_sampled(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step, const void* draft_logits,
                         const float* row_lse_in, uint64_t seed, uint64_t cycle, float* row_lse,
                         int32_t* frontier_tokens, int32_t* frontier_count, void* stream) {
    EAGLE_CALL(stream, ws);
    const uint64_t sc[2] = {seed, cycle};
    return expand_call(cfg, ws, ws_bytes, step, draft_logits, row_lse_in, row_lse, frontier_tokens, frontier_count,
                       stream, false, sc);
}

int eagle_test_expand_starved(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step,
                              const void* draft_logits, float* row_lse, int32_t* frontier_tokens,
                              int32_t* frontier_count, void* stream) {
    EAGLE_CALL(stream, ws);
    return expand_call(cfg, ws, ws_bytes, step, draft_logits, nullptr, row_lse, frontier_tokens, frontier_count,
                       stream, true);
}

int eagle_lmhead(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int hidden_dim, const void* hidden,
                 const void* weight, void* draft_logits, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (!hidden || !weight || !draft_logits || hidden_dim < 8) return EAGLE_ERR_INVALID_ARG;
    if (hidden_dim % 8 != 0 || !aligned16(hidden) || !aligned16(weight) || !aligned16(draft_logits))
        return EAGLE_ERR_UNSUPPORTED;
    return launch_result(launch_lmhead(d.B * d.k, d.V, hidden_dim, hidden, weight, d.dtype, draft_logits, w.status,
                                       static_cast<cudaStream_t>(stream)));
}

size_t eagle_lmhead_topk_scratch_bytes(const eagle_tree_cfg* cfg) {
    TreeDims d;
    if (resolve(cfg, &d) != EAGLE_OK) return 0;
    return lmhead_topk_scratch_bytes(static_cast<long>(d.B) * d.k, d.k);
}

int eagle_lmhead_topk(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int hidden_dim, const void* hidden,
                      const void* weight, void* scratch, size_t scratch_bytes, float* row_lse, int32_t* topk_ids,
                      float* topk_logits, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (!hidden || !weight || !row_lse || !topk_ids || !topk_logits || hidden_dim < 8) return EAGLE_ERR_INVALID_ARG;
    if (hidden_dim % 8 != 0 || !aligned16(hidden) || !aligned16(weight)) return EAGLE_ERR_UNSUPPORTED;
    const long M = static_cast<long>(d.B) * d.k;
    if (M > 4096) return EAGLE_ERR_UNSUPPORTED;
    if (scratch == nullptr || (reinterpret_cast<uintptr_t>(scratch) & 255u) != 0 ||
        scratch_bytes < lmhead_topk_scratch_bytes(M, d.k))
        return EAGLE_ERR_WORKSPACE;
    return launch_result(launch_lmhead_topk(static_cast<int>(M), d.V, hidden_dim, d.k, hidden, weight, d.dtype,
                                            scratch, row_lse, topk_ids, topk_logits, w.status,
                                            static_cast<cudaStream_t>(stream)));
}

int eagle_rerank(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    return launch_result(launch_rerank(d, w, static_cast<cudaStream_t>(stream)));
}

int eagle_tree_value(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, float* value_sum, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (value_sum == nullptr) return EAGLE_ERR_INVALID_ARG;
    return launch_result(launch_tree_value(d, w, value_sum, static_cast<cudaStream_t>(stream)));
}

int eagle_build_tree(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, const int32_t* prefix_len,
                     const int32_t* root_token, int32_t* tokens, int32_t* parent, int32_t* depth, int32_t* pos_ids,
                     uint32_t* mask, int32_t* n_tree, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (!prefix_len || !root_token || !tokens || !parent || !depth || !pos_ids || !mask || !n_tree)
        return EAGLE_ERR_INVALID_ARG;
    return launch_result(launch_build_tree(d, w, prefix_len, root_token, tokens, parent, depth, pos_ids, mask, n_tree,
                                           static_cast<cudaStream_t>(stream)));
}

size_t eagle_attention_workspace_bytes(const eagle_kv_cfg* kv, int T) {
    KvDims k;
    if (resolve_kv(kv, &k) != EAGLE_OK || T < 1 || T > kMaxSlots) return 0;
    return attention_ws_bytes(k, T);
}

int eagle_tree_attention(const eagle_kv_cfg* kv, int T, const void* q, const void* kv_cache, int layer,
                         const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out, void* ws,
                         size_t ws_bytes, void* stream) {
    EAGLE_CALL(stream, ws);
    KvDims k;
    int rc = resolve_kv(kv, &k);
    if (rc != EAGLE_OK) return rc;
    if (T < 1 || T > kMaxSlots || layer < 0) return EAGLE_ERR_INVALID_ARG;
    if (!q || !kv_cache || !prefix_len || !mask || !n_tree || !out) return EAGLE_ERR_INVALID_ARG;
    if (k.d > 128) return EAGLE_ERR_UNSUPPORTED;
    const size_t need = attention_ws_bytes(k, T);
    if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return EAGLE_ERR_WORKSPACE;
    return launch_result(launch_attention(k, T, q, kv_cache, layer, prefix_len, mask, n_tree, out, ws, ws_bytes,
                                          static_cast<int*>(ws), static_cast<cudaStream_t>(stream)));
}

int eagle_verify(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int mode, float temperature, uint64_t seed,
                 uint64_t cycle, const void* target_logits, const void* draft_logits, const int32_t* tokens,
                 const int32_t* parent, const int32_t* n_tree, int32_t* accept_len, int32_t* accepted_slots,
                 int32_t* out_tokens, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (mode != EAGLE_VERIFY_GREEDY && mode != EAGLE_VERIFY_LOSSLESS && mode != EAGLE_VERIFY_DRAFT)
        return EAGLE_ERR_INVALID_ARG;
    if (!target_logits || !tokens || !parent || !n_tree || !accept_len || !accepted_slots || !out_tokens)
        return EAGLE_ERR_INVALID_ARG;
    if (mode == EAGLE_VERIFY_DRAFT && draft_logits == nullptr) return EAGLE_ERR_INVALID_ARG;
    float inv_t = 1.0f;
    if (mode != EAGLE_VERIFY_GREEDY) {
        if (!(temperature > 0.0f) || !std::isfinite(temperature)) return EAGLE_ERR_INVALID_ARG;
        inv_t = static_cast<float>(1.0 / static_cast<double>(temperature));
    }
    if (!aligned16(target_logits)) return EAGLE_ERR_UNSUPPORTED;
    if (mode == EAGLE_VERIFY_DRAFT)
        return launch_result(launch_verify_draft(d, w, inv_t, verify_rng(seed, cycle), target_logits, draft_logits,
                                                 tokens, parent, n_tree, accept_len, accepted_slots, out_tokens,
                                                 static_cast<cudaStream_t>(stream)));
    return launch_result(launch_verify(d, w, mode, inv_t, target_logits, tokens, parent, n_tree,
                                       verify_rng(seed, cycle), accept_len, accepted_slots, out_tokens,
                                       static_cast<cudaStream_t>(stream)));
}

int eagle_shard_partials(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int rows, int shard_vocab,
                         int vocab_offset, const void* logits, float* part_max_sum, uint64_t* part_keys,
                         void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (!logits || !part_max_sum || !part_keys || rows < 1 || rows > 65535 || shard_vocab < 1 || vocab_offset < 0 ||
        static_cast<long>(vocab_offset) + shard_vocab > d.V)
        return EAGLE_ERR_INVALID_ARG;
    const int esize = d.dtype == EAGLE_BF16 ? 2 : 4;
    if ((static_cast<long>(shard_vocab) * esize) % 16 != 0 || !aligned16(logits)) return EAGLE_ERR_UNSUPPORTED;
    return launch_result(launch_shard_partials(shard_vocab, d.k, rows, d.dtype, logits, vocab_offset,
                                               reinterpret_cast<float2*>(part_max_sum), part_keys, w.status,
                                               static_cast<cudaStream_t>(stream)));
}

int eagle_shard_merge(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int n_shards, int rows,
                      const float* part_max_sum, const uint64_t* part_keys, float* row_lse, int32_t* topk_ids,
                      float* topk_logits, int32_t* row_argmax, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (!part_max_sum || !part_keys || !row_lse || !topk_ids || !topk_logits || !row_argmax || rows < 1 ||
        n_shards < 1)
        return EAGLE_ERR_INVALID_ARG;
    if (n_shards > kShardMax) return EAGLE_ERR_UNSUPPORTED;
    return launch_result(launch_shard_merge(n_shards, rows, d.k, reinterpret_cast<const float2*>(part_max_sum),
                                            part_keys, row_lse, topk_ids, topk_logits, row_argmax, w.status,
                                            static_cast<cudaStream_t>(stream)));
}

int eagle_expand_topk(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, int step, const int32_t* topk_ids,
                      const float* topk_logits, const float* row_lse_in, float* row_lse, int32_t* frontier_tokens,
                      int32_t* frontier_count, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (step < 0 || step >= d.D) return EAGLE_ERR_INVALID_ARG;
    if (!topk_ids || !topk_logits || !row_lse_in || !row_lse || !frontier_tokens || !frontier_count)
        return EAGLE_ERR_INVALID_ARG;
    return launch_result(launch_expand_topk(d, w, step, topk_ids, topk_logits, row_lse_in, row_lse, frontier_tokens,
                                            frontier_count, static_cast<cudaStream_t>(stream)));
}

int eagle_verify_argmax(const eagle_tree_cfg* cfg, void* ws, size_t ws_bytes, const int32_t* row_argmax,
                        const int32_t* tokens, const int32_t* parent, const int32_t* n_tree, int32_t* accept_len,
                        int32_t* accepted_slots, int32_t* out_tokens, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    if (!row_argmax || !tokens || !parent || !n_tree || !accept_len || !accepted_slots || !out_tokens)
        return EAGLE_ERR_INVALID_ARG;
    return launch_result(launch_verify_argmax(d, w, row_argmax, tokens, parent, n_tree, accept_len, accepted_slots,
                                              out_tokens, static_cast<cudaStream_t>(stream)));
}

int eagle_kv_compact(const eagle_kv_cfg* kv, void* kv_cache, const int32_t* prefix_len, const int32_t* accept_len,
                     const int32_t* accepted_slots, int slots_stride, int32_t* new_len, void* ws, void* stream) {
    EAGLE_CALL(stream, ws);
    KvDims k;
    int rc = resolve_kv(kv, &k);
    if (rc != EAGLE_OK) return rc;
    if (!kv_cache || !prefix_len || !accept_len || !accepted_slots || !new_len || slots_stride < 1)
        return EAGLE_ERR_INVALID_ARG;
    const int esize = k.dtype == EAGLE_BF16 ? 2 : 4;
    if ((static_cast<int64_t>(k.Hkv) * k.d * esize) % 16 != 0 || (k.pos_stride * esize) % 16 != 0 ||
        (k.seq_stride * esize) % 16 != 0 || (k.layer_stride * esize) % 16 != 0 || (k.kv_stride * esize) % 16 != 0 ||
        !aligned16(kv_cache))
        return EAGLE_ERR_UNSUPPORTED;
    if (k.layers == 0) return EAGLE_OK;
    if (k.layers * 2 > 65535) return EAGLE_ERR_UNSUPPORTED;
    return launch_result(launch_kv_compact(k, kv_cache, prefix_len, accept_len, accepted_slots, slots_stride, new_len,
                                           static_cast<int*>(ws), static_cast<cudaStream_t>(stream)));
}

int eagle_status_fetch(void* ws, int* device_status, void* stream) {
    if (ws == nullptr || device_status == nullptr) return EAGLE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return EAGLE_ERR_LAUNCH;
    int v = 0;
    if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return EAGLE_ERR_LAUNCH;
    if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return EAGLE_ERR_LAUNCH;
    *device_status = v;
    if (v == 0) return EAGLE_OK;
    return v == 2 ? EAGLE_ERR_TIMEOUT : EAGLE_ERR_DEVICE;
}

int eagle_tree_export(const eagle_tree_cfg* cfg, const void* ws, size_t ws_bytes, int32_t* cand_token,
                      int32_t* cand_parent, int32_t* cand_depth, float* cand_logv, uint8_t* cand_valid, uint8_t* kept,
                      int32_t* n_kept, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t BC = static_cast<size_t>(d.B) * d.C;
    cudaError_t e = cudaSuccess;
    auto cp = [&](void* dst, const void* src, size_t bytes) {
        if (dst && e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
    };
    cp(cand_token, w.cand_token, BC * 4);
    cp(cand_parent, w.cand_parent, BC * 4);
    cp(cand_depth, w.cand_depth, BC * 4);
    cp(cand_logv, w.cand_logv, BC * 4);
    cp(cand_valid, w.cand_valid, BC);
    cp(kept, w.kept, BC);
    cp(n_kept, w.n_kept, static_cast<size_t>(d.B) * 4);
    return launch_result(e);
}

int eagle_verify_export(const eagle_tree_cfg* cfg, const void* ws, size_t ws_bytes, float* row_max,
                        int32_t* row_argmax, uint64_t* row_mass, void* stream) {
    EAGLE_CALL(stream, ws);
    TreeDims d;
    TreeWs w;
    int rc = resolve(cfg, &d);
    if (rc == EAGLE_OK) rc = bind_ws(d, ws, ws_bytes, &w);
    if (rc != EAGLE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t BT = static_cast<size_t>(d.B) * d.T;
    cudaError_t e = cudaSuccess;
    auto cp = [&](void* dst, const void* src, size_t bytes) {
        if (dst && e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
    };
    cp(row_max, w.row_max, BT * 4);
    cp(row_argmax, w.row_arg, BT * 4);
    cp(row_mass, w.row_mass, BT * 8);
    return launch_result(e);
}

int eagle_test_sampling(const uint32_t* words, const float* ys, int n, float* gumbel_out, float* log_out,
                        void* stream) {
    EAGLE_CALL(stream, nullptr);
    if (n < 0 || (words && !gumbel_out) || (ys && !log_out)) return EAGLE_ERR_INVALID_ARG;
    if (n == 0) return EAGLE_OK;
    return launch_result(launch_sampling_probe(words, ys, n, gumbel_out, log_out, static_cast<cudaStream_t>(stream)));
}

uint64_t eagle_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int eagle_last_cuda_error(const char** message) {
    const int e = g_last_cuda_error;
    if (message) *message = e ? cudaGetErrorString(static_cast<cudaError_t>(e)) : "no error";
    return e;
}

const char* eagle_status_string(int status) {
    switch (status) {
        case EAGLE_OK: return "ok";
        case EAGLE_ERR_INVALID_ARG: return "invalid argument";
        case EAGLE_ERR_UNSUPPORTED: return "unsupported configuration";
        case EAGLE_ERR_LAUNCH: return "CUDA launch or runtime error";
        case EAGLE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case EAGLE_ERR_DEVICE: return "device reported a fault";
        case EAGLE_ERR_TIMEOUT: return "device wait gave up";
        default: return "unknown status";
    }
}

}  // extern "C"
