// CPU oracle for the EAGLE-2 dynamic draft-tree cycle.
//
// TEST INFRASTRUCTURE ONLY. This file is a plain, slow, single-threaded
// statement of what each stage of the cycle computes. It is called by the
// tests, by the package's smoke check and by the benchmark's CPU-baseline leg,
// and by nothing on the product path. It shares no code, header, table or
// constant generator with the CUDA library; inputs come from the separate
// seeded generator module.
//
// Sources (page title and section):
//  [EAGLE-2 summary]  "EAGLE-2: Faster Inference of Language Models with
//                      Dynamic Draft Trees" (paperlayer summary of arXiv
//                      2406.16858v2): 2.1 Speculative Sampling, 4.1 Expansion
//                      Phase, 4.2 Reranking Phase, App. A.
//  [Dynamic trees]    "EAGLE-2: Dynamic Draft Trees" (stable-lab tutorial):
//                      "Value of a Node = Its Path Product", "Common
//                      misconception".
//  [EAGLE notes]      "EAGLE" (garden.houmin.site, Chinese notes): EAGLE 方法
//                      (TopK drafting, tree attention), EAGLE 2 方法 (Expand /
//                      ReRank with threshold and tie rule).
//
// Where the pages are silent the plain reading is taken; each such reading is
// named at the function that uses it.
//
// Parity status of each function (what pins it is in the CPU test-suite):
//   row_stats, expand, rerank, build_tree, attention, verify_greedy,
//   verify_lossless, kv_compact, dexp, value_sum, lmhead_logits,
//   expand_sampled, dlog, gumbel, verify_draft: pinned (closed forms, library
//   routines, brute force, the tutorial's worked chain, one-hot rows and a
//   float64 matmul for the LM head, chi-square against the sampling and
//   target distributions for sampled drafting).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------- inputs ---

// Logit element -> float. dtype 0 = fp32, 1 = bf16 (upper half of an fp32).
float load_logit(const void* base, int dtype, int64_t idx) {
    if (dtype == 0) return static_cast<const float*>(base)[idx];
    uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(base)[idx]) << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return f;
}

// Candidate node numbering used throughout: step s (0-based) expands up to k
// frontier nodes, each into k children, so step s owns ids
// [base(s), base(s) + k*k) with base(0) = 0 (one frontier node: the root) and
// base(s) = k + (s-1) k^2. Child id = base(s) + f*k + r for frontier slot f and
// child rank r. Ids are therefore depth-major.
int64_t step_base(int s, int k) { return s == 0 ? 0 : k + static_cast<int64_t>(s - 1) * k * k; }

// ------------------------------------------------------ stage 1: a draft row ---

// Softmax statistics and top-k of one vocabulary row [EAGLE notes, EAGLE 方法:
// TopK drafting over the LM-head distribution]. lse = m + log(sum exp(x - m)) in
// double, rounded once to float. Top-k ranks by (logit desc, token id asc): the
// pages do not order equal logits, the lower id is taken first.
void row_stats(const void* row, int dtype, int V, int k, double* lse64, std::vector<int>* topk) {
    double m = -INFINITY;
    for (int x = 0; x < V; ++x) m = std::max(m, static_cast<double>(load_logit(row, dtype, x)));
    double s = 0.0;
    for (int x = 0; x < V; ++x) s += std::exp(static_cast<double>(load_logit(row, dtype, x)) - m);
    *lse64 = m + std::log(s);
    std::vector<int> ids(V);
    for (int x = 0; x < V; ++x) ids[x] = x;
    int kk = std::min(k, V);
    std::partial_sort(ids.begin(), ids.begin() + kk, ids.end(), [&](int a, int b) {
        float xa = load_logit(row, dtype, a), xb = load_logit(row, dtype, b);
        if (xa != xb) return xa > xb;
        return a < b;
    });
    topk->assign(ids.begin(), ids.begin() + kk);
}

// Fixed-order exp used by lossless verification so that CPU and GPU reach the
// same integer probabilities. Written from the mathematics: Cody-Waite
// reduction z = n ln2 + r with ln2 split into a 16-bit head and a tail, a
// degree-7 Taylor polynomial of exp(r) in Horner form, then scaling by 2^n.
// Every step is one correctly rounded fp32 operation: n is z log2(e) rounded
// to the nearest integer (ties to even) by one fused multiply-add with
// 1.5 * 2^23, the reduction and each Horner step are fused multiply-adds
// (std::fma), the scaling is exact. No other contraction (built with
// -ffp-contract=off). Defined for z <= 0; returns 0 below -32.
float dexp(float z) {
    if (!(z >= -32.0f)) return 0.0f;
    const float kLog2e = 1.44269502f;             // 0x3FB8AA3B
    const float kLn2Hi = 0.693145751953125f;      // 0x3F317200, 16 significant bits
    const float kLn2Lo = 1.42860677e-06f;         // 0x35BFBE8E = ln2 - kLn2Hi
    const float kRound = 12582912.0f;             // 1.5 * 2^23
    const float t = std::fma(z, kLog2e, kRound);  // kRound + nearest integer to z log2(e)
    const float n = t - kRound;                   // exact
    float r = std::fma(-n, kLn2Hi, z);
    r = std::fma(-n, kLn2Lo, r);
    const float c[8] = {1.0f, 1.0f, 0.5f, 1.0f / 6.0f, 1.0f / 24.0f, 1.0f / 120.0f, 1.0f / 720.0f,
                        1.0f / 5040.0f};
    float p = c[7];
    for (int i = 6; i >= 0; --i) p = std::fma(p, r, c[i]);
    const int e = static_cast<int>(n) + 127;
    uint32_t sb = static_cast<uint32_t>(e) << 23;
    float scale;
    std::memcpy(&scale, &sb, 4);
    return p * scale;
}

// Integer probability mass of token x in a row with maximum m at inverse
// temperature inv_t: floor(dexp((x - m) * inv_t) * 2^40).
uint64_t fixed_mass(float x, float m, float inv_t) {
    float z = (x - m) * inv_t;
    float e = dexp(z);
    return static_cast<uint64_t>(e * 1099511627776.0f);  // exact: power-of-two scale, then floor
}

// Fixed-order natural logarithm of a positive normal float, for the Gumbel
// keys of sampled drafting; every step is one correctly rounded fp32
// operation so that another implementation of the same steps reaches the
// same bits (reading: a sampled child is an integer decided by floating
// point, so both sides take it in the same precision). Written from the
// mathematics: y = m 2^e with m in [sqrt(1/2), sqrt(2)) (exact bit
// operations), s = (m - 1) / (m + 1), ln m = 2 atanh(s) = 2 s (1 + s^2/3 +
// s^4/5 + s^6/7 + s^8/9 + s^10/11) in Horner form in s^2 by fused
// multiply-adds (the next term is below 2^-33 relative for |s| <= 0.172),
// then ln y = e ln2_hi + (e ln2_lo + ln m) with the 16-bit head of ln 2 used
// by dexp (e ln2_hi exact).
float dlog(float y) {
    uint32_t b;
    std::memcpy(&b, &y, 4);
    int e = static_cast<int>((b >> 23) & 0xffu) - 127;
    const uint32_t mb = (b & 0x7fffffu) | 0x3f800000u;
    float m;
    std::memcpy(&m, &mb, 4);
    if (m > 1.41421353816986083984375f) {  // fp32 just below sqrt(2)
        m = m * 0.5f;
        e += 1;
    }
    const float s = (m - 1.0f) / (m + 1.0f);
    const float z = s * s;
    float p = 1.0f / 11.0f;
    p = std::fmaf(p, z, 1.0f / 9.0f);
    p = std::fmaf(p, z, 1.0f / 7.0f);
    p = std::fmaf(p, z, 1.0f / 5.0f);
    p = std::fmaf(p, z, 1.0f / 3.0f);
    p = std::fmaf(p, z, 1.0f);
    float t = s * p;
    t = t + t;
    const float ef = static_cast<float>(e);
    return std::fmaf(ef, 0.693145751953125f, std::fmaf(ef, 1.42860677e-06f, t));
}

// Gumbel noise of a 32-bit uniform word: u = ((w >> 9) + 1/2) 2^-23, exact in
// fp32 and strictly inside (0, 1); g = -ln(-ln u) by dlog.
float gumbel_of_word(uint32_t w) {
    const float u = (static_cast<float>(w >> 9) + 0.5f) * 0x1p-23f;
    return -dlog(-dlog(u));
}

// The k children of one row drawn from q = softmax(row) without replacement,
// in drawing order: the k largest keys fl(x + g(w_x)) (the Gumbel-top-k
// identity: perturbing log-probabilities by independent Gumbel noise and
// sorting gives sequential sampling without replacement); equal keys go to
// the lower id. NaN entries are never drawn.
void sampled_topk(const void* row, int dtype, int V, int k, const uint32_t* words, std::vector<int>* out) {
    std::vector<std::pair<float, int>> keys;
    keys.reserve(V);
    for (int x = 0; x < V; ++x) {
        const float v = load_logit(row, dtype, x);
        if (v != v) continue;
        keys.emplace_back(v + gumbel_of_word(words[x]), x);
    }
    const int kk = std::min<int>(k, static_cast<int>(keys.size()));
    std::partial_sort(keys.begin(), keys.begin() + kk, keys.end(), [](const auto& a, const auto& c) {
        if (a.first != c.first) return a.first > c.first;
        return a.second < c.second;
    });
    out->clear();
    for (int i = 0; i < kk; ++i) out->push_back(keys[i].second);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- stage 1 ---

// One row: lse (double and its float rounding) and the top-k token ids.
int oracle_row_stats(const void* row, int dtype, int V, int k, double* lse64_out, float* lse_out,
                     int32_t* topk_out) {
    double lse64;
    std::vector<int> topk;
    row_stats(row, dtype, V, k, &lse64, &topk);
    *lse64_out = lse64;
    *lse_out = static_cast<float>(lse64);
    for (int r = 0; r < static_cast<int>(topk.size()); ++r) topk_out[r] = topk[r];
    return 0;
}

float oracle_dexp(float z) { return dexp(z); }

// -------------------------------------------------------- tree state reset ---

// Candidate table [B, C]: token, parent (node id, -1 = root), depth, logv,
// valid. Frontier [B, k] node ids (-1 = root) and count [B].
void oracle_tree_init(int B, int C, int k, int32_t* cand_token, int32_t* cand_parent,
                      int32_t* cand_depth, float* cand_logv, uint8_t* cand_valid, int32_t* fnode,
                      int32_t* fcount) {
    for (int64_t i = 0; i < static_cast<int64_t>(B) * C; ++i) {
        cand_token[i] = -1;
        cand_parent[i] = -1;
        cand_depth[i] = -1;
        cand_logv[i] = -INFINITY;
        cand_valid[i] = 0;
    }
    for (int b = 0; b < B; ++b) {
        for (int f = 0; f < k; ++f) fnode[b * k + f] = -1;
        fcount[b] = 1;  // the root is the only frontier node of step 0
    }
}

// ------------------------------------------------------ stages 1+2: expand ---

// One expansion step s for every sequence.
//
// Each frontier node f of sequence b owns draft row logits_s[b, f, :]. Its k
// highest-logit tokens become its children [EAGLE notes, EAGLE 方法: each draft
// token gets its own children, not a Cartesian product]. A child's value is
// the product of confidences on its root path [Dynamic trees, "Value of a Node
// = Its Path Product"; EAGLE-2 summary 4.1: the confidence c_j stands in for
// the acceptance rate], held as a log: logv(child) = logv(parent) + (x - lse),
// both fp32 operations, logv(root) = 0.
//
// The next frontier is the top-k of this step's children by value [EAGLE-2
// summary 4.1: expand the top-k nodes of the current layer], taken only among
// children whose value is at least the threshold [EAGLE notes, EAGLE 2 方法,
// Expand: a node whose path probability is below the threshold is not
// expanded]. Reading: threshold compared in the log domain (log_thr is passed
// in, -inf = off); equal values rank by lower node id.
//
// lse_in: if non-null, the row lse values [B, k] to use instead of this
// oracle's own (stage-chained parity runs feed the GPU's fp32 lse here).
//
// policy 1 (ablation "confidence-based expansion", EAGLE-2 summary 5.2.1:
// value-based expansion compared with confidence-based): the next frontier is
// ranked by the child's own confidence lp = x - lse instead of its value; the
// threshold still applies to the value. cand_lp [B, C] receives lp.
//
// policy 3 (the EAGLE-1 static shape that the tutorial's widget sets against
// the dynamic tree, "Watch the Budget Being Spent": the same branching
// pattern for every context): the next frontier is chosen by position only,
// child r of frontier slot f ranked by f + r ascending, then by lower node id
// (reading: a fixed triangular pattern that favours the first children of
// the first slots, as a hand-shaped tree does).
static int expand_impl(int B, int V, int k, int step, int dtype, float log_thr, int policy, const void* logits_s,
                       const float* lse_in, const uint32_t* words_s, int C, int32_t* cand_token,
                       int32_t* cand_parent, int32_t* cand_depth, float* cand_logv, float* cand_lp,
                       uint8_t* cand_valid, int32_t* fnode, int32_t* fcount, float* row_lse_out, int32_t* ftok_out,
                       int32_t* fcount_out) {
    const int64_t base = step_base(step, k);
    for (int b = 0; b < B; ++b) {
        const int F = fcount[b];
        for (int f = 0; f < F; ++f) {
            const int64_t row_off = (static_cast<int64_t>(b) * k + f) * V;
            const void* row = dtype == 0
                                  ? static_cast<const void*>(static_cast<const float*>(logits_s) + row_off)
                                  : static_cast<const void*>(static_cast<const uint16_t*>(logits_s) + row_off);
            double lse64;
            std::vector<int> topk;
            row_stats(row, dtype, V, k, &lse64, &topk);
            if (words_s) sampled_topk(row, dtype, V, k, words_s + row_off, &topk);
            float lse = lse_in ? lse_in[b * k + f] : static_cast<float>(lse64);
            if (row_lse_out) row_lse_out[b * k + f] = lse;
            const int parent = fnode[b * k + f];
            const float plogv = parent < 0 ? 0.0f : cand_logv[static_cast<int64_t>(b) * C + parent];
            for (int r = 0; r < static_cast<int>(topk.size()); ++r) {
                const int64_t id = base + static_cast<int64_t>(f) * k + r;
                if (id >= C) return -1;
                const int64_t at = static_cast<int64_t>(b) * C + id;
                float x = load_logit(row, dtype, topk[r]);
                float lp = x - lse;
                cand_token[at] = topk[r];
                cand_parent[at] = parent;
                cand_depth[at] = step + 1;
                cand_logv[at] = plogv + lp;
                cand_lp[at] = lp;
                cand_valid[at] = 1;
            }
        }
        // Next frontier: eligible children of this step, best first.
        std::vector<int> elig;
        for (int f = 0; f < F; ++f)
            for (int r = 0; r < k; ++r) {
                int id = static_cast<int>(base + static_cast<int64_t>(f) * k + r);
                int64_t at = static_cast<int64_t>(b) * C + id;
                if (cand_valid[at] && cand_logv[at] >= log_thr) elig.push_back(id);
            }
        if (policy == 3) {
            auto pos = [&](int id) {
                const int i = static_cast<int>(id - base);
                return i / k + i % k;
            };
            std::sort(elig.begin(), elig.end(), [&](int a, int c) {
                if (pos(a) != pos(c)) return pos(a) < pos(c);
                return a < c;
            });
        } else {
            const float* rank_by = policy == 1 ? cand_lp : cand_logv;
            std::sort(elig.begin(), elig.end(), [&](int a, int c) {
                float va = rank_by[static_cast<int64_t>(b) * C + a];
                float vc = rank_by[static_cast<int64_t>(b) * C + c];
                if (va != vc) return va > vc;
                return a < c;
            });
        }
        const int nf = std::min<int>(k, static_cast<int>(elig.size()));
        for (int f = 0; f < k; ++f) {
            fnode[b * k + f] = f < nf ? elig[f] : -1;
            if (ftok_out)
                ftok_out[b * k + f] = f < nf ? cand_token[static_cast<int64_t>(b) * C + elig[f]] : -1;
        }
        fcount[b] = nf;
        if (fcount_out) fcount_out[b] = nf;
    }
    return 0;
}

int oracle_expand(int B, int V, int k, int step, int dtype, float log_thr, int policy, const void* logits_s,
                  const float* lse_in, int C, int32_t* cand_token, int32_t* cand_parent,
                  int32_t* cand_depth, float* cand_logv, float* cand_lp, uint8_t* cand_valid, int32_t* fnode,
                  int32_t* fcount, float* row_lse_out, int32_t* ftok_out, int32_t* fcount_out) {
    return expand_impl(B, V, k, step, dtype, log_thr, policy, logits_s, lse_in, nullptr, C, cand_token, cand_parent,
                       cand_depth, cand_logv, cand_lp, cand_valid, fnode, fcount, row_lse_out, ftok_out, fcount_out);
}

// Sampled drafting (next row f4: children drawn from the draft distribution
// instead of its top-k, so that the draft-probability acceptance rule can be
// used; reading: Gumbel-top-k over per-element uniform words [B, k, V] of
// the step, values and everything after the draw exactly as oracle_expand).
int oracle_expand_sampled(int B, int V, int k, int step, int dtype, float log_thr, int policy,
                          const void* logits_s, const float* lse_in, const uint32_t* words_s, int C,
                          int32_t* cand_token, int32_t* cand_parent, int32_t* cand_depth, float* cand_logv,
                          float* cand_lp, uint8_t* cand_valid, int32_t* fnode, int32_t* fcount, float* row_lse_out,
                          int32_t* ftok_out, int32_t* fcount_out) {
    if (!words_s) return -1;
    return expand_impl(B, V, k, step, dtype, log_thr, policy, logits_s, lse_in, words_s, C, cand_token, cand_parent,
                       cand_depth, cand_logv, cand_lp, cand_valid, fnode, fcount, row_lse_out, ftok_out, fcount_out);
}

int oracle_dlog(int n, const float* y, float* out) {
    for (int i = 0; i < n; ++i) out[i] = dlog(y[i]);
    return 0;
}

int oracle_gumbel(int n, const uint32_t* w, float* out) {
    for (int i = 0; i < n; ++i) out[i] = gumbel_of_word(w[i]);
    return 0;
}

// --------------------------------------------------------- stage 3: rerank ---

// Keep the N most valuable candidates of all drafted tokens [EAGLE-2 summary
// 4.2: rerank all draft tokens, keep the top m by value; EAGLE notes, EAGLE 2
// 方法, ReRank: on equal values the shallower node is kept]. Ties beyond depth
// go to the lower node id (reading). Full sort, then the first min(N, #valid).
//
// policy 2 (ablation "without reranking", EAGLE-2 summary 5.2.2): the
// candidates are only the nodes chosen by the expansion phase, i.e. the
// frontier of every step 1..D (fhist [D+1, B, k], -1 = none; reading: these
// are the tokens drafted without a rerank, k per depth), of which the first N
// by the same order are kept.
//
// policy 3 (static shape): the same candidates as policy 2, the first N by
// depth, then lower node id: a shape that does not depend on the values.
int oracle_rerank(int B, int C, int N, int policy, int D, int k, const int32_t* fhist, const int32_t* cand_depth,
                  const float* cand_logv, const uint8_t* cand_valid, uint8_t* kept, int32_t* n_kept) {
    for (int b = 0; b < B; ++b) {
        std::vector<int> ids;
        if (policy == 2 || policy == 3) {
            for (int s = 1; s <= D; ++s)
                for (int f = 0; f < k; ++f) {
                    const int id = fhist[(static_cast<int64_t>(s) * B + b) * k + f];
                    if (id >= 0 && cand_valid[static_cast<int64_t>(b) * C + id]) ids.push_back(id);
                }
        } else {
            for (int i = 0; i < C; ++i)
                if (cand_valid[static_cast<int64_t>(b) * C + i]) ids.push_back(i);
        }
        std::sort(ids.begin(), ids.end(), [&](int a, int c) {
            int64_t ia = static_cast<int64_t>(b) * C + a, ic = static_cast<int64_t>(b) * C + c;
            if (policy != 3 && cand_logv[ia] != cand_logv[ic]) return cand_logv[ia] > cand_logv[ic];
            if (cand_depth[ia] != cand_depth[ic]) return cand_depth[ia] < cand_depth[ic];
            return a < c;
        });
        const int n = std::min<int>(N, static_cast<int>(ids.size()));
        for (int i = 0; i < C; ++i) kept[static_cast<int64_t>(b) * C + i] = 0;
        for (int j = 0; j < n; ++j) kept[static_cast<int64_t>(b) * C + ids[j]] = 1;
        n_kept[b] = n;
    }
    return 0;
}

// ------------------------------------------------------ stage 4: emission ---

// Flatten the kept tree [EAGLE-2 summary 4.2: the selected tokens are
// flattened into a one-dimensional sequence with an attention mask that keeps
// branches apart; EAGLE notes, EAGLE 方法: tree attention verifies every
// branch in one pass]. Reading: slot 0 is the root (the last verified token),
// slots 1..n are the kept nodes in node-id order (depth-major, so parents come
// before children). Mask row i = ancestors-or-self of slot i, bit j of word
// j/32 (LSB first). Position id = prefix_len + depth. Unused slots are -1 with
// zero mask rows. Returns -2 if a kept node's parent is not kept.
int oracle_build_tree(int B, int C, int T, int W, const int32_t* prefix_len,
                      const int32_t* root_token, const int32_t* cand_token,
                      const int32_t* cand_parent, const int32_t* cand_depth,
                      const uint8_t* kept, int32_t* tokens, int32_t* parent, int32_t* depth,
                      int32_t* pos, uint32_t* mask, int32_t* n_tree, int32_t* slot_of) {
    for (int b = 0; b < B; ++b) {
        int32_t* tk = tokens + static_cast<int64_t>(b) * T;
        int32_t* pa = parent + static_cast<int64_t>(b) * T;
        int32_t* de = depth + static_cast<int64_t>(b) * T;
        int32_t* po = pos + static_cast<int64_t>(b) * T;
        uint32_t* mk = mask + static_cast<int64_t>(b) * T * W;
        int32_t* so = slot_of + static_cast<int64_t>(b) * C;
        for (int i = 0; i < T; ++i) {
            tk[i] = pa[i] = de[i] = po[i] = -1;
            for (int w = 0; w < W; ++w) mk[i * W + w] = 0;
        }
        tk[0] = root_token[b];
        de[0] = 0;
        po[0] = prefix_len[b];
        mk[0] = 1u;
        int n = 1;
        for (int id = 0; id < C; ++id) {
            int64_t at = static_cast<int64_t>(b) * C + id;
            so[id] = -1;
            if (!kept[at]) continue;
            if (n >= T) return -3;
            int ps = 0;
            if (cand_parent[at] >= 0) {
                ps = so[cand_parent[at]];
                if (ps < 0) return -2;
            }
            so[id] = n;
            tk[n] = cand_token[at];
            pa[n] = ps;
            de[n] = cand_depth[at];
            po[n] = prefix_len[b] + cand_depth[at];
            for (int w = 0; w < W; ++w) mk[n * W + w] = mk[ps * W + w];
            mk[n * W + n / 32] |= 1u << (n % 32);
            ++n;
        }
        n_tree[b] = n;
    }
    return 0;
}

// Expected number of accepted tokens approximated by the summed value of the
// kept nodes [Dynamic trees, "Value of a Node = Its Path Product":
// E[#accepted] ~ sum over the tree of Value(v)], in double.
double oracle_value_sum(int C, const float* cand_logv, const uint8_t* kept) {
    double s = 0.0;
    for (int i = 0; i < C; ++i)
        if (kept[i]) s += std::exp(static_cast<double>(cand_logv[i]));
    return s;
}

// ------------------------------------------------ stage 5: tree attention ---

// Tree-masked attention of one (sequence b, slot i, query head h) row
// [EAGLE notes, EAGLE 方法: Medusa-style tree attention; EAGLE-2 summary 4.2].
// Keys: every prefix position [0, L_b) plus the tree slots j whose bit is set
// in mask row i (stored at cache position L_b + j). Scale 1/sqrt(d); query
// head h reads KV head h / (Hq/Hkv). Dot products, softmax and the weighted
// sum in double over the widened inputs. out[d] receives the result; rows
// i >= n_tree are zero.
//
// q: [B, T, Hq, d]; k_base/v_base: element (b, pos, hkv, e) at
// b*seq_stride + pos*pos_stride + hkv*d + e.
void attention_row(int T, int Hq, int Hkv, int d, int dtype, const void* q, const void* k_base,
                   const void* v_base, int64_t seq_stride, int64_t pos_stride,
                   const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, int W,
                   int b, int i, int h, double* out) {
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (i >= n_tree[b]) return;
    const int L = prefix_len[b];
    const int hk = h / (Hq / Hkv);
    std::vector<int64_t> keys;
    for (int p = 0; p < L; ++p) keys.push_back(p);
    for (int j = 0; j < T; ++j)
        if (mask[(static_cast<int64_t>(b) * T + i) * W + j / 32] >> (j % 32) & 1u) keys.push_back(L + j);
    const int64_t qoff = ((static_cast<int64_t>(b) * T + i) * Hq + h) * d;
    std::vector<double> qv(d);
    for (int e = 0; e < d; ++e) qv[e] = load_logit(q, dtype, qoff + e);
    const double scale = 1.0 / std::sqrt(static_cast<double>(d));
    std::vector<double> sc(keys.size());
    double mx = -INFINITY;
    for (size_t t = 0; t < keys.size(); ++t) {
        int64_t koff = b * seq_stride + keys[t] * pos_stride + static_cast<int64_t>(hk) * d;
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += qv[e] * static_cast<double>(load_logit(k_base, dtype, koff + e));
        sc[t] = dot * scale;
        mx = std::max(mx, sc[t]);
    }
    double den = 0.0;
    for (size_t t = 0; t < keys.size(); ++t) {
        sc[t] = std::exp(sc[t] - mx);
        den += sc[t];
    }
    for (size_t t = 0; t < keys.size(); ++t) {
        int64_t voff = b * seq_stride + keys[t] * pos_stride + static_cast<int64_t>(hk) * d;
        double w = sc[t] / den;
        for (int e = 0; e < d; ++e) out[e] += w * static_cast<double>(load_logit(v_base, dtype, voff + e));
    }
}

// All rows: out [B, T, Hq, d] doubles.
void oracle_attention(int B, int T, int Hq, int Hkv, int d, int dtype, const void* q,
                      const void* k_base, const void* v_base, int64_t seq_stride,
                      int64_t pos_stride, const int32_t* prefix_len, const uint32_t* mask,
                      const int32_t* n_tree, int W, double* out) {
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < T; ++i)
            for (int h = 0; h < Hq; ++h)
                attention_row(T, Hq, Hkv, d, dtype, q, k_base, v_base, seq_stride, pos_stride,
                              prefix_len, mask, n_tree, W, b, i, h,
                              out + ((static_cast<int64_t>(b) * T + i) * Hq + h) * d);
}

// Selected rows only (sampled checks at full size): rows[3*r..] = (b, i, h).
void oracle_attention_rows(int n_rows, const int32_t* rows, int T, int Hq, int Hkv, int d,
                           int dtype, const void* q, const void* k_base, const void* v_base,
                           int64_t seq_stride, int64_t pos_stride, const int32_t* prefix_len,
                           const uint32_t* mask, const int32_t* n_tree, int W, double* out) {
    for (int r = 0; r < n_rows; ++r)
        attention_row(T, Hq, Hkv, d, dtype, q, k_base, v_base, seq_stride, pos_stride, prefix_len,
                      mask, n_tree, W, rows[3 * r], rows[3 * r + 1], rows[3 * r + 2],
                      out + static_cast<int64_t>(r) * d);
}

// ---------------------------------------------------------- stage 6: verify ---

namespace {

int row_argmax(const void* row, int dtype, int V) {
    int best = 0;
    float bv = load_logit(row, dtype, 0);
    for (int x = 1; x < V; ++x) {
        float v = load_logit(row, dtype, x);
        if (v > bv) {  // strict: equal logits keep the lower id
            bv = v;
            best = x;
        }
    }
    return best;
}

const void* row_ptr(const void* base, int dtype, int64_t row, int V) {
    return dtype == 0 ? static_cast<const void*>(static_cast<const float*>(base) + row * V)
                      : static_cast<const void*>(static_cast<const uint16_t*>(base) + row * V);
}

void write_path(int b, int Dp1, int a, const int* path, const int32_t* tk, int bonus,
                int32_t* accept_len, int32_t* accepted_slots, int32_t* out_tokens) {
    accept_len[b] = a;
    for (int j = 0; j < Dp1; ++j) {
        accepted_slots[b * Dp1 + j] = j <= a ? path[j] : -1;
        out_tokens[b * Dp1 + j] = j < a ? tk[path[j + 1]] : j == a ? bonus : -1;
    }
}

}  // namespace

// Greedy verification [EAGLE-2 summary 2.1: the target scores every draft
// token and tokens are accepted in order]: at temperature 0 the target's
// choice at slot t is argmax of target row t (equal logits: lower id). From
// the root, move to the child whose token equals the target's choice at the
// current slot; stop when there is none. Output: accepted count a, slots of
// the path (root first), the a accepted tokens followed by the target's choice
// at the last path slot (the bonus token).
int oracle_verify_greedy(int B, int T, int V, int Dp1, int dtype, const void* target,
                         const int32_t* tokens, const int32_t* parent, const int32_t* n_tree,
                         int32_t* accept_len, int32_t* accepted_slots, int32_t* out_tokens,
                         int32_t* argmax_out) {
    for (int b = 0; b < B; ++b) {
        const int n = n_tree[b];
        const int32_t* tk = tokens + static_cast<int64_t>(b) * T;
        const int32_t* pa = parent + static_cast<int64_t>(b) * T;
        std::vector<int> g(T, -1);
        for (int t = 0; t < n; ++t) g[t] = row_argmax(row_ptr(target, dtype, static_cast<int64_t>(b) * T + t, V), dtype, V);
        if (argmax_out)
            for (int t = 0; t < T; ++t) argmax_out[b * T + t] = g[t];
        std::vector<int> path(1, 0);
        int cur = 0;
        for (;;) {
            int next = -1;
            for (int c = 1; c < n; ++c)
                if (pa[c] == cur && tk[c] == g[cur]) {
                    next = c;
                    break;
                }
            if (next < 0 || static_cast<int>(path.size()) >= Dp1) break;
            path.push_back(next);
            cur = next;
        }
        write_path(b, Dp1, static_cast<int>(path.size()) - 1, path.data(), tk, g[cur], accept_len,
                   accepted_slots, out_tokens);
    }
    return 0;
}

// Lossless verification [EAGLE-2 summary 2.1 and abstract: tokens are
// accepted sequentially by the probability ratio and the output distribution
// is unchanged]. The draft children are the deterministic top-k of the draft
// row, so the proposal of a tested child x is a point mass; the ratio rule
// min(1, p/q) then accepts x with probability p_cur(x), and a rejection
// removes x from p_cur (residual max(0, p - q) renormalised). Reading: at node
// u, the kept children are tested in slot order; the first accepted child
// becomes the new node (p reset to its own target row); if none is accepted,
// or u has no kept child, the bonus token is drawn from the residual p_cur.
//
// Probabilities are integers so both implementations agree exactly:
// P[x] = floor(dexp((x - m) * inv_t) * 2^40) with m the row maximum; S = sum P.
// Uniforms are inputs: u[b, c] (word) tests the child at slot c with
// U24 = u >> 8, accept iff U24 * S_cur < 2^24 * P[x]; the draw uses
// U64 = u[b, T+1] * 2^32 + u[b, T], t = floor(U64 * S_cur / 2^64) and takes the
// smallest token y not removed whose running sum of P exceeds t.
int oracle_verify_lossless(int B, int T, int V, int Dp1, int dtype, float inv_t, const void* target,
                           const int32_t* tokens, const int32_t* parent, const int32_t* n_tree,
                           const uint32_t* uniforms, int32_t* accept_len, int32_t* accepted_slots,
                           int32_t* out_tokens, float* row_max_out, uint64_t* row_mass_out) {
    std::vector<uint64_t> P(V);
    for (int b = 0; b < B; ++b) {
        const int n = n_tree[b];
        const int32_t* tk = tokens + static_cast<int64_t>(b) * T;
        const int32_t* pa = parent + static_cast<int64_t>(b) * T;
        const uint32_t* u = uniforms + static_cast<int64_t>(b) * (T + 2);
        if (row_max_out || row_mass_out)
            for (int t = 0; t < T; ++t) {
                float m = -INFINITY;
                uint64_t S = 0;
                if (t < n) {
                    const void* row = row_ptr(target, dtype, static_cast<int64_t>(b) * T + t, V);
                    for (int x = 0; x < V; ++x) m = std::max(m, load_logit(row, dtype, x));
                    for (int x = 0; x < V; ++x) S += fixed_mass(load_logit(row, dtype, x), m, inv_t);
                }
                if (row_max_out) row_max_out[b * T + t] = m;
                if (row_mass_out) row_mass_out[b * T + t] = S;
            }
        std::vector<int> path(1, 0);
        int cur = 0;
        int bonus = -1;
        for (;;) {
            const void* row = row_ptr(target, dtype, static_cast<int64_t>(b) * T + cur, V);
            float m = -INFINITY;
            for (int x = 0; x < V; ++x) m = std::max(m, load_logit(row, dtype, x));
            uint64_t S = 0;
            for (int x = 0; x < V; ++x) {
                P[x] = fixed_mass(load_logit(row, dtype, x), m, inv_t);
                S += P[x];
            }
            std::vector<char> removed(V, 0);
            int next = -1;
            for (int c = 1; c < n && static_cast<int>(path.size()) < Dp1; ++c) {
                if (pa[c] != cur) continue;
                const int x = tk[c];
                const unsigned __int128 lhs = static_cast<unsigned __int128>(u[c] >> 8) * S;
                const unsigned __int128 rhs = static_cast<unsigned __int128>(P[x]) << 24;
                if (lhs < rhs) {
                    next = c;
                    break;
                }
                S -= P[x];
                removed[x] = 1;
            }
            if (next >= 0) {
                path.push_back(next);
                cur = next;
                continue;
            }
            const uint64_t U64 = (static_cast<uint64_t>(u[T + 1]) << 32) | u[T];
            const uint64_t t = static_cast<uint64_t>((static_cast<unsigned __int128>(U64) * S) >> 64);
            uint64_t run = 0;
            for (int y = 0; y < V; ++y) {
                if (removed[y]) continue;
                run += P[y];
                if (run > t) {
                    bonus = y;
                    break;
                }
            }
            break;
        }
        write_path(b, Dp1, static_cast<int>(path.size()) - 1, path.data(), tk, bonus, accept_len,
                   accepted_slots, out_tokens);
    }
    return 0;
}

// Verification with the draft-probability rule (next row f4) [EAGLE-2
// summary 2.1: tokens accepted sequentially by the probability ratio]. At
// node u with target p_cur and draft q_cur (the softmax of the row u's
// children were drawn from, without replacement and in slot order), child x
// is accepted with probability min(1, p_cur(x) / q_cur(x)); on rejection
// p_cur becomes the residual max(0, p_cur - q_cur) renormalised and x leaves
// q_cur (renormalised: the next child was drawn without it). The first
// accepted child becomes the new node (p and q reset to its own rows); if
// none is accepted, or u has no kept child, the bonus token is drawn from
// p_cur. This is the target distribution exactly when the tested children
// of every node are its drawn children in drawing order (a token-independent
// tree shape); a tree kept by draft value is not (reading, pinned by exact
// enumeration and by sampling in the tests).
//
// Integer arithmetic in the style of oracle_verify_lossless: P and Q are
// fixed_mass integers (2^40 scale) of the target and draft rows, A the
// current target residual with sum SA, Q with sum SQ. Child x (uniform word
// u[b, c] of its slot c, U24 = u >> 8) is accepted iff
// U24 * Q[x] * SA < 2^24 * A[x] * SQ. A rejection sets
// r(y) = max(0, A[y] * SQ - Q[y] * SA) (the residual scaled by SA * SQ) and
// A = floor(r / 2^s), s the smallest shift that brings max r to 2^40 or
// below (A is kept when every r is 0); then SQ -= Q[x], Q[x] = 0. The bonus
// draw is the lossless one on A: t = floor(U64 * SA / 2^64), the smallest y
// whose running sum of A exceeds t.
//   draft      [R, V] draft rows; draft_row [B, T] row of the slot's node
//              (-1: never expanded, then the node has no kept child).
int oracle_verify_draft(int B, int T, int V, int Dp1, int dtype, float inv_t, const void* target,
                        const void* draft, const int64_t* draft_row, const int32_t* tokens, const int32_t* parent,
                        const int32_t* n_tree, const uint32_t* uniforms, int32_t* accept_len,
                        int32_t* accepted_slots, int32_t* out_tokens) {
    typedef unsigned __int128 u128;
    std::vector<uint64_t> A(V), Q(V);
    std::vector<u128> r(V);
    for (int b = 0; b < B; ++b) {
        const int n = n_tree[b];
        const int32_t* tk = tokens + static_cast<int64_t>(b) * T;
        const int32_t* pa = parent + static_cast<int64_t>(b) * T;
        const uint32_t* u = uniforms + static_cast<int64_t>(b) * (T + 2);
        std::vector<int> path(1, 0);
        int cur = 0;
        int bonus = -1;
        for (;;) {
            const void* prow = row_ptr(target, dtype, static_cast<int64_t>(b) * T + cur, V);
            float m = -INFINITY;
            for (int x = 0; x < V; ++x) m = std::max(m, load_logit(prow, dtype, x));
            uint64_t SA = 0;
            for (int x = 0; x < V; ++x) {
                A[x] = fixed_mass(load_logit(prow, dtype, x), m, inv_t);
                SA += A[x];
            }
            const int64_t dr = draft_row[static_cast<int64_t>(b) * T + cur];
            uint64_t SQ = 0;
            if (dr >= 0) {
                const void* qrow = row_ptr(draft, dtype, dr, V);
                float mq = -INFINITY;
                for (int x = 0; x < V; ++x) mq = std::max(mq, load_logit(qrow, dtype, x));
                for (int x = 0; x < V; ++x) {
                    Q[x] = fixed_mass(load_logit(qrow, dtype, x), mq, inv_t);
                    SQ += Q[x];
                }
            }
            int next = -1;
            for (int c = 1; c < n && static_cast<int>(path.size()) < Dp1; ++c) {
                if (pa[c] != cur) continue;
                if (dr < 0) return -2;  // a kept child of a node that was never expanded
                const int x = tk[c];
                const u128 lhs = static_cast<u128>(static_cast<uint64_t>(u[c] >> 8) * Q[x]) * SA;
                const u128 rhs = (static_cast<u128>(A[x]) * SQ) << 24;
                if (lhs < rhs) {
                    next = c;
                    break;
                }
                u128 mx = 0;
                for (int y = 0; y < V; ++y) {
                    const u128 pa_ = static_cast<u128>(A[y]) * SQ, qa = static_cast<u128>(Q[y]) * SA;
                    r[y] = pa_ > qa ? pa_ - qa : 0;
                    mx = std::max(mx, r[y]);
                }
                if (mx > 0) {
                    int sh = 0;
                    while ((mx >> sh) > (static_cast<u128>(1) << 40)) ++sh;
                    SA = 0;
                    for (int y = 0; y < V; ++y) {
                        A[y] = static_cast<uint64_t>(r[y] >> sh);
                        SA += A[y];
                    }
                }
                SQ -= Q[x];
                Q[x] = 0;
            }
            if (next >= 0) {
                path.push_back(next);
                cur = next;
                continue;
            }
            const uint64_t U64 = (static_cast<uint64_t>(u[T + 1]) << 32) | u[T];
            const uint64_t t = static_cast<uint64_t>((static_cast<u128>(U64) * SA) >> 64);
            uint64_t run = 0;
            for (int y = 0; y < V; ++y) {
                run += A[y];
                if (run > t) {
                    bonus = y;
                    break;
                }
            }
            break;
        }
        write_path(b, Dp1, static_cast<int>(path.size()) - 1, path.data(), tk, bonus, accept_len, accepted_slots,
                   out_tokens);
    }
    return 0;
}

// -------------------------------------------------------- stage 6b: compact ---

// Move the accepted path's KV into the contiguous cache (not on the pages;
// the plain reading of "compaction of the accepted nodes' KV"): for every
// layer and for K and V, position L_b + j receives what position
// L_b + accepted_slots[b, j] held before the call, j = 1..a. All sources are
// read before any destination is written. new_len = L_b + a + 1 (the root at
// L_b stays; the bonus token has no KV yet).
//
// cache: bytes; element (b, layer, kv, pos, h, e) at
// b*seq_stride + layer*layer_stride + kv*kv_stride + pos*pos_stride + h*d + e.
int oracle_kv_compact(int B, int layers, int Hkv, int d, int elem_size, void* cache,
                      int64_t seq_stride, int64_t layer_stride, int64_t kv_stride,
                      int64_t pos_stride, const int32_t* prefix_len, const int32_t* accept_len,
                      const int32_t* accepted_slots, int Dp1, int32_t* new_len) {
    const int64_t row_bytes = static_cast<int64_t>(Hkv) * d * elem_size;
    char* base = static_cast<char*>(cache);
    for (int b = 0; b < B; ++b) {
        const int a = accept_len[b];
        const int L = prefix_len[b];
        for (int l = 0; l < layers; ++l)
            for (int kv = 0; kv < 2; ++kv) {
                char* region = base + (b * seq_stride + l * layer_stride + kv * kv_stride) * elem_size;
                std::vector<char> tmp(static_cast<size_t>(a) * row_bytes);
                for (int j = 1; j <= a; ++j)
                    std::memcpy(tmp.data() + (j - 1) * row_bytes,
                                region + (L + accepted_slots[b * Dp1 + j]) * pos_stride * elem_size, row_bytes);
                for (int j = 1; j <= a; ++j)
                    std::memcpy(region + (L + j) * pos_stride * elem_size, tmp.data() + (j - 1) * row_bytes,
                                row_bytes);
            }
        new_len[b] = L + a + 1;
    }
    return 0;
}


// ------------------------------------------------ LM head (next row f1) ---

// Logits of M frontier rows through the LM head, the step before stage 1
// ["EAGLE" notes, EAGLE 方法: the draft model reuses the target's LM head;
// reading: logits[m, v] = sum_h hidden[m, h] * W[v, h] with bf16 hidden
// states [M, H] and weights [V, H] (row v holds vocabulary entry v), each
// product exact in double, summed in double in h order and rounded once to
// float]. Stage 1 then runs on these fp32 rows.
int oracle_lmhead_logits(int M, int V, int H, const uint16_t* hidden, const uint16_t* W, float* logits) {
    if (M < 0 || V < 1 || H < 1) return -1;
    std::vector<double> hrow(static_cast<size_t>(H));
    for (int m = 0; m < M; ++m) {
        for (int h = 0; h < H; ++h) hrow[h] = load_logit(hidden, 1, static_cast<int64_t>(m) * H + h);
        for (int v = 0; v < V; ++v) {
            const uint16_t* wr = W + static_cast<int64_t>(v) * H;
            double s = 0.0;
            for (int h = 0; h < H; ++h) s += hrow[h] * static_cast<double>(load_logit(wr, 1, h));
            logits[static_cast<int64_t>(m) * V + v] = static_cast<float>(s);
        }
    }
    return 0;
}

}  // extern "C"
