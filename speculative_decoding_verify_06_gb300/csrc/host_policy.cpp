// host_policy.cpp -- host-side companions of the verify pass: the depth policy and the n-gram
// drafter.  No GPU work; they read what svd_accept wrote and feed drafts to the next pass.
//
// "Decode is memory-bound ...", sections "Speculative decoding" and "Two things the math says
// to do": with i.i.d. acceptance alpha, a pass at depth k yields (1 - alpha^(k+1)) / (1 - alpha)
// tokens, and counting the drafter (one draft step costs c of a target pass) the speedup is
// that over (k c + 1); the fork's --spec-adapt throttles the depth when the measured
// acceptance falls below 35 %.
// "100 tokens per second ...", section "Lever 3: an n-gram overlay for repetition": an
// incremental map from the last L tokens to whatever followed them last time, over the prompt
// and everything generated; a hit proposes that continuation as drafts (L = 6 won the sweep).
#include <cmath>
#include <cstdint>
#include <unordered_map>
#include <vector>

#include "svd.h"

namespace {

double expected_tokens(double alpha, int k) {
    if (alpha >= 1.0) return (double)(k + 1);
    if (alpha <= 0.0) return 1.0;
    return (1.0 - std::pow(alpha, k + 1)) / (1.0 - alpha);
}

double speedup(double alpha, int k, double c) { return expected_tokens(alpha, k) / (k * c + 1.0); }

int best_depth(double alpha, double c, int k_max) {
    int best = 1;
    double sb = speedup(alpha, 1, c);
    for (int k = 2; k <= k_max; ++k) {
        const double s = speedup(alpha, k, c);
        if (s > sb) {  // ties keep the shallower depth
            sb = s;
            best = k;
        }
    }
    return best;
}

}  // namespace

struct svd_spec_adapt {
    int k_max;
    double cost, threshold, decay;
    double accepted = 0.0, trials = 0.0;  // decayed counts
};

struct svd_ngram {
    int L;
    uint64_t base_pow;  // B^(L-1)
    std::vector<int32_t> hist;
    uint64_t roll = 0;  // hash of the last L tokens once hist.size() >= L
    // hash of a key -> continuation start of the latest occurrence of each distinct key with
    // that hash (a key is compared token by token, so collisions never return a wrong hit)
    std::unordered_map<uint64_t, std::vector<int64_t>> map;
};

namespace {
constexpr uint64_t kHashBase = 0x9E3779B97F4A7C15ull;

bool same_key(const svd_ngram *g, int64_t end_a, int64_t end_b) {
    for (int i = 1; i <= g->L; ++i)
        if (g->hist[end_a - i] != g->hist[end_b - i]) return false;
    return true;
}
}  // namespace

extern "C" {

double svd_expected_tokens_per_pass(double alpha, int k) {
    if (k < 0 || !(alpha >= 0.0 && alpha <= 1.0)) return NAN;
    return expected_tokens(alpha, k);
}

double svd_speedup(double alpha, int k, double draft_cost) {
    if (k < 0 || !(alpha >= 0.0 && alpha <= 1.0) || !(draft_cost >= 0.0)) return NAN;
    return speedup(alpha, k, draft_cost);
}

int svd_best_depth(double alpha, double draft_cost, int k_max) {
    if (k_max < 1 || !(alpha >= 0.0 && alpha <= 1.0) || !(draft_cost >= 0.0)) return SVD_ERR_INVALID_ARG;
    return best_depth(alpha, draft_cost, k_max);
}

svd_spec_adapt *svd_spec_adapt_create(int k_max, double draft_cost, double threshold,
                                      double half_life_windows) {
    if (k_max < 1 || k_max > SVD_K_MAX || !(draft_cost >= 0.0) || !(threshold >= 0.0 && threshold <= 1.0) ||
        !(half_life_windows > 0.0))
        return nullptr;
    svd_spec_adapt *a = new svd_spec_adapt;
    a->k_max = k_max;
    a->cost = draft_cost;
    a->threshold = threshold;
    a->decay = std::pow(0.5, 1.0 / half_life_windows);
    return a;
}

int svd_spec_adapt_observe(svd_spec_adapt *a, const int32_t *n_emitted, const int32_t *status,
                           int64_t n_windows, int k) {
    if (!a || (!n_emitted && n_windows > 0) || n_windows < 0 || k < 1) return SVD_ERR_INVALID_ARG;
    for (int64_t w = 0; w < n_windows; ++w) {
        if (status && status[w] != 0) continue;  // a window with bad inputs says nothing
        const int ne = n_emitted[w];
        if (ne < 1 || ne > k + 1) continue;
        const int j = ne - 1;  // drafts accepted; a rejection followed unless all k were
        a->accepted = a->accepted * a->decay + j;
        a->trials = a->trials * a->decay + j + (j < k ? 1 : 0);
    }
    return SVD_OK;
}

double svd_spec_adapt_alpha(const svd_spec_adapt *a) {
    if (!a || a->trials <= 0.0) return NAN;
    return a->accepted / a->trials;
}

int svd_spec_adapt_depth(const svd_spec_adapt *a) {
    if (!a) return SVD_ERR_INVALID_ARG;
    if (a->trials <= 0.0) return a->k_max;  // nothing measured yet
    const double alpha = a->accepted / a->trials;
    if (alpha < a->threshold) return 1;  // depth buys almost nothing here
    return best_depth(alpha, a->cost, a->k_max);
}

void svd_spec_adapt_destroy(svd_spec_adapt *a) { delete a; }

svd_ngram *svd_ngram_create(int key_len) {
    if (key_len < 1 || key_len > 64) return nullptr;
    svd_ngram *g = new svd_ngram;
    g->L = key_len;
    g->base_pow = 1;
    for (int i = 1; i < key_len; ++i) g->base_pow *= kHashBase;
    return g;
}

int svd_ngram_append(svd_ngram *g, const int32_t *tokens, int64_t n) {
    if (!g || n < 0 || (!tokens && n > 0)) return SVD_ERR_INVALID_ARG;
    const int L = g->L;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t m = (int64_t)g->hist.size();  // index of the new token
        // the key ending just before the new token now has a continuation: record it
        if (m >= L) {
            std::vector<int64_t> &bucket = g->map[g->roll];
            bool found = false;
            for (int64_t &p : bucket)
                if (same_key(g, p, m)) {
                    p = m;
                    found = true;
                    break;
                }
            if (!found) bucket.push_back(m);
        }
        const uint32_t t = (uint32_t)tokens[i];
        if (m >= L) g->roll -= (uint64_t)(uint32_t)g->hist[m - L] * g->base_pow;
        g->roll = g->roll * kHashBase + t;
        g->hist.push_back(tokens[i]);
    }
    return SVD_OK;
}

int svd_ngram_propose(const svd_ngram *g, int32_t *out, int k_max) {
    if (!g || k_max < 0 || (!out && k_max > 0)) return SVD_ERR_INVALID_ARG;
    const int64_t n = (int64_t)g->hist.size();
    if (n < g->L || k_max == 0) return 0;
    const auto it = g->map.find(g->roll);
    if (it == g->map.end()) return 0;
    for (const int64_t p : it->second) {
        if (!same_key(g, p, n)) continue;
        const int64_t cnt = std::min<int64_t>(k_max, n - p);
        for (int64_t i = 0; i < cnt; ++i) out[i] = g->hist[p + i];
        return (int)cnt;
    }
    return 0;
}

int64_t svd_ngram_length(const svd_ngram *g) { return g ? (int64_t)g->hist.size() : -1; }

void svd_ngram_destroy(svd_ngram *g) { delete g; }

}  // extern "C"
