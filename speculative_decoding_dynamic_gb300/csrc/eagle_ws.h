// Workspace layout and launcher declarations shared by the host entry points
// and the kernel files of libeagle. Internal; not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace eagle {

constexpr int kMaxTopK = 16;
constexpr int kMaxDepth = 16;
constexpr int kMaxSlots = 256;       // T = N + 1
constexpr int kMaxCandidates = 1024;  // C = k + (D-1) k^2
constexpr int kMaxChunks = 8;        // CTAs per logit row (one thread-block cluster)

// Row kernels: a CTA's segment of a logit row moves through shared memory in
// chunks of kRowChunkBytes (one bulk copy each), at most kRowStages chunks
// resident at once; kRowWarpsPerCta consumer warps each own 1/8 of a chunk.
constexpr int kRowChunkBytes = 16384;
constexpr int kRowStages = 4;
constexpr int kRowWarpsPerCta = 8;

// Elements of a row segment when the row is split over `cpr` CTAs (a multiple
// of 16 bytes, so every segment starts on a 16-byte boundary).
inline int row_seg_elems(int V, int esize, int cpr) {
    const int epv = 16 / esize;
    const int seg = (V + cpr - 1) / cpr;
    return (seg + epv - 1) / epv * epv;
}
inline int row_chunks(int seg, int esize) { return (seg * esize + kRowChunkBytes - 1) / kRowChunkBytes; }

// Resolved problem description passed by value to kernels.
struct TreeDims {
    int B, V, k, D, N, T, W, C;
    float log_thr;  // -inf disables the threshold
    int dtype;      // 0 fp32, 1 bf16
    int policy;     // 0 EAGLE-2, 1 confidence-based expansion, 2 without rerank
};

// Pointers into the caller's workspace. Layout computed by ws_layout(). The
// status word is always the first word of a workspace (tree or attention).
struct TreeWs {
    int* status;            // [1] first-error-wins device status
    int* expand_ticket;     // [B] arrivals of row clusters in the current expand step
    int* verify_ticket;     // [B] arrivals of row clusters in verify
    int32_t* cand_token;    // [B, C]
    int32_t* cand_parent;   // [B, C] node id of the parent, -1 = root
    int32_t* cand_depth;    // [B, C]
    float* cand_logv;       // [B, C] log path value
    float* cand_lp;         // [B, C] the node's own log-probability (confidence)
    uint8_t* cand_valid;    // [B, C]
    int32_t* fnode;         // [D+1, B, k] frontier node ids per step (-1 = root)
    int32_t* fcount;        // [D+1, B]
    uint8_t* kept;          // [B, C]
    int32_t* n_kept;        // [B]
    int32_t* slot_of;       // [B, C] tree slot of a kept node, -1 otherwise
    float* row_max;         // [B, T] verify row maximum
    int32_t* row_arg;       // [B, T] verify row argmax
    uint64_t* row_mass;     // [B, T] verify integer mass
    uint64_t* pmass;        // [B, T] lossless: integer mass of slot c's token in its parent's row
    uint64_t* resid;        // [B, V] target residual of the draft-probability rule
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Computes the layout; returns total bytes. If base != nullptr fills ws.
inline size_t ws_layout(const TreeDims& d, void* base, TreeWs* ws) {
    size_t off = 0;
    char* p = static_cast<char*>(base);
    auto take = [&](size_t bytes) -> void* {
        off = align_up(off, 256);
        void* r = p ? static_cast<void*>(p + off) : nullptr;
        off += bytes;
        return r;
    };
    const size_t B = d.B, C = d.C, k = d.k, D = d.D, T = d.T;
    TreeWs w{};
    w.status = static_cast<int*>(take(sizeof(int)));
    w.expand_ticket = static_cast<int*>(take(B * sizeof(int)));
    w.verify_ticket = static_cast<int*>(take(B * sizeof(int)));
    w.cand_token = static_cast<int32_t*>(take(B * C * 4));
    w.cand_parent = static_cast<int32_t*>(take(B * C * 4));
    w.cand_depth = static_cast<int32_t*>(take(B * C * 4));
    w.cand_logv = static_cast<float*>(take(B * C * 4));
    w.cand_lp = static_cast<float*>(take(B * C * 4));
    w.cand_valid = static_cast<uint8_t*>(take(B * C));
    w.fnode = static_cast<int32_t*>(take((D + 1) * B * k * 4));
    w.fcount = static_cast<int32_t*>(take((D + 1) * B * 4));
    w.kept = static_cast<uint8_t*>(take(B * C));
    w.n_kept = static_cast<int32_t*>(take(B * 4));
    w.slot_of = static_cast<int32_t*>(take(B * C * 4));
    w.row_max = static_cast<float*>(take(B * T * 4));
    w.row_arg = static_cast<int32_t*>(take(B * T * 4));
    w.row_mass = static_cast<uint64_t*>(take(B * T * 8));
    w.pmass = static_cast<uint64_t*>(take(B * T * 8));
    w.resid = static_cast<uint64_t*>(take(B * static_cast<size_t>(d.V) * 8));
    if (ws) *ws = w;
    return align_up(off, 256);
}

// How a logit row is split over a thread-block cluster and streamed.
struct RowPlan {
    int cpr;     // CTAs per row (cluster size), power of two <= kMaxChunks
    int seg;     // elements per CTA (row_seg_elems); the last CTA may get fewer
    int nch;     // chunks per full segment
    int stages;  // shared-memory stages (all nch when the segment stays resident)
    int smem;    // dynamic shared memory per CTA
};
// rows = logit rows of the launch.
RowPlan plan_rows(int V, int esize, long rows, int max_stages, int max_seg_chunks);

// ----------------------------------------------------------- launchers ---
// Each returns cudaSuccess or the launch error. All enqueue on `stream`.
cudaError_t launch_tree_init(const TreeDims& d, const TreeWs& ws, cudaStream_t stream);
// starve_ring: the failure-path test hook (the row ring's producer issues no
// copies, so the consumers' bounded waits give up and raise status 2).
// sample_seed_cycle: {seed, cycle} for sampled drafting (children drawn from
// the row's softmax without replacement), NULL for the top-k children.
cudaError_t launch_expand(const TreeDims& d, const TreeWs& ws, int step, const void* logits, const float* lse_in,
                          float* row_lse, int32_t* ftok, int32_t* fcount_out, cudaStream_t stream,
                          bool starve_ring = false, const uint64_t* sample_seed_cycle = nullptr);
cudaError_t launch_rerank(const TreeDims& d, const TreeWs& ws, cudaStream_t stream);
cudaError_t launch_tree_value(const TreeDims& d, const TreeWs& ws, float* value_sum, cudaStream_t stream);
cudaError_t launch_build_tree(const TreeDims& d, const TreeWs& ws, const int32_t* prefix_len,
                              const int32_t* root_token, int32_t* tokens, int32_t* parent, int32_t* depth,
                              int32_t* pos, uint32_t* mask, int32_t* n_tree, cudaStream_t stream);
// Counter-based uniforms of lossless verification: word c of sequence b is
// word 0 of Philox4x32-10 at counter (c, b, c2, c3) under key (k0, k1), where
// (k0, k1) = (seed_lo ^ kVerifyStream, seed_hi) and (c2, c3) = (cycle_lo, cycle_hi).
constexpr uint32_t kVerifyStream = 7;
struct VerifyRng {
    uint32_t k0, k1, c2, c3;
};
inline VerifyRng verify_rng(uint64_t seed, uint64_t cycle) {
    return VerifyRng{static_cast<uint32_t>(seed) ^ kVerifyStream, static_cast<uint32_t>(seed >> 32),
                     static_cast<uint32_t>(cycle), static_cast<uint32_t>(cycle >> 32)};
}
cudaError_t launch_verify(const TreeDims& d, const TreeWs& ws, int mode, float inv_temp, const void* target,
                          const int32_t* tokens, const int32_t* parent, const int32_t* n_tree, VerifyRng rng,
                          int32_t* accept_len, int32_t* slots, int32_t* out_tokens, cudaStream_t stream);
// Lossless acceptance walk (after launch_verify's row statistics): one
// cluster per sequence; the integer masses of the rows it visits only.
cudaError_t launch_verify_walk(const TreeDims& d, const TreeWs& ws, float inv_temp, VerifyRng rng, const void* target,
                               const int32_t* tokens, const int32_t* parent, const int32_t* n_tree,
                               int32_t* accept_len, int32_t* slots, int32_t* out_tokens, cudaStream_t stream);

// Vocabulary slices: stage-1 partials of `rows` rows of a slice [rows, Vs]
// (keys carry token id id_base + index), their merge over S slices, stage 2
// from merged top-k, and the greedy walk from merged argmax.
constexpr int kShardMax = 16;
cudaError_t launch_shard_partials(int Vs, int k, int rows, int dtype, const void* logits, int id_base, float2* part_ms,
                                  uint64_t* part_keys, int* status, cudaStream_t stream);
cudaError_t launch_shard_merge(int S, int rows, int k, const float2* part_ms, const uint64_t* part_keys, float* lse,
                               int32_t* topk_id, float* topk_val, int32_t* argmax, int* status, cudaStream_t stream);
cudaError_t launch_expand_topk(const TreeDims& d, const TreeWs& ws, int step, const int32_t* topk_id,
                               const float* topk_val, const float* lse_in, float* row_lse, int32_t* ftok,
                               int32_t* fcount_out, cudaStream_t stream);
cudaError_t launch_verify_argmax(const TreeDims& d, const TreeWs& ws, const int32_t* row_argmax, const int32_t* tokens,
                                 const int32_t* parent, const int32_t* n_tree, int32_t* accept_len, int32_t* slots,
                                 int32_t* out_tokens, cudaStream_t stream);

cudaError_t launch_verify_draft(const TreeDims& d, const TreeWs& ws, float inv_temp, VerifyRng rng,
                                const void* target, const void* draft, const int32_t* tokens, const int32_t* parent,
                                const int32_t* n_tree, int32_t* accept_len, int32_t* slots, int32_t* out_tokens,
                                cudaStream_t stream);
cudaError_t launch_sampling_probe(const uint32_t* words, const float* ys, int n, float* gumbel_out, float* log_out,
                                  cudaStream_t stream);

struct KvDims {
    int B, Hq, Hkv, d, layers, max_len, dtype;
    int64_t seq_stride, layer_stride, kv_stride, pos_stride;
};
cudaError_t launch_kv_compact(const KvDims& kv, void* cache, const int32_t* prefix_len, const int32_t* accept_len,
                              const int32_t* slots, int slots_stride, int32_t* new_len, int* status,
                              cudaStream_t stream);

size_t attention_ws_bytes(const KvDims& kv, int T);
// The persistent two-CTA-per-SM attention pipeline (k_attn_pipe.cu) serves
// shapes whose unsplit items fill two CTAs on every SM.
bool attention_pipe_fits(const KvDims& kv, int T);
cudaError_t launch_attention_pipe(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                                  const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                                  int* status, cudaStream_t stream);
// LM-head logits [M, V] (fp32, or bf16 when out_dtype is 1) of hidden [M, H]
// and weight [V, H] (bf16), on the tensor cores.
cudaError_t launch_lmhead(int M, int V, int H, const void* hidden, const void* weight, int out_dtype, void* out,
                          int* status, cudaStream_t stream);
// The same product with stage 1 in the epilogue: the logits are rounded to
// out_dtype as launch_lmhead would store them but never leave the SM; each
// epilogue thread keeps a running (max, sum of exp, top-k keys) of one row
// over its CTA's vocabulary tiles, writes it to `scratch` once, and a merge
// gives the row's lse and top-k. scratch holds lmhead_topk_scratch_bytes(M, k)
// bytes (256-byte aligned); M <= 4096.
constexpr int kLmShards = 160;  // most CTAs of the fused launch (>= SMs of the GPU)
size_t lmhead_topk_scratch_bytes(long M, int k);
cudaError_t launch_lmhead_topk(int M, int V, int H, int k, const void* hidden, const void* weight, int out_dtype,
                               void* scratch, float* row_lse, int32_t* topk_id, float* topk_val, int* status,
                               cudaStream_t stream);
cudaError_t launch_attention(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                             const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                             void* ws, size_t ws_bytes, int* status, cudaStream_t stream);

// Raise a kernel's dynamic shared memory limit on the current device when a
// launch needs more than was set before (no attribute call once set, so that
// launches inside a stream capture that follow a first call make none).
cudaError_t ensure_dyn_smem(const void* kernel, int smem);

// Host-side launch counter (incremented by every launcher).
void count_launch(int n = 1);

// Launch with programmatic stream serialisation (see pdl_wait_prior).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launch();
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace eagle
