// tree_build.cpp -- the greedy sparse candidate tree (host code).
//
// "Speculative-Decoding / Medusa" blog, section 四 (optimized tree
// construction): with a_k^(i) the accuracy of head k's i-th ranked token,
// taken as independent, the node reached by the rank path [i_1 .. i_m] is
// accepted with probability prod_j a_j^(i_j); E[L] sums that product over the
// tree's nodes; the tree grows from the root one node at a time, always by the
// candidate (a child of a node already in the tree) of largest product, up to
// a fixed node count.
//
// A max-heap holds exactly the candidates: the children of every chosen node
// that are not chosen yet.  A child's product is its parent's times one more
// factor, which is the left-to-right product from 1 along the path.  Equal
// products go to the smaller depth, then to the lexicographically smaller rank
// path.  The chosen nodes are numbered by (depth, rank path), so every parent
// precedes its children and the array feeds spec_tree_mask and
// spec_verify_tree as it is.  Runs on the host: a few dozen nodes, built once
// per accuracy table, not per decode step.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <map>
#include <queue>
#include <vector>

#include "host.h"
#include "spec_verify.h"

namespace spec {
namespace {

struct Cand {
    double v;
    std::vector<int> path;  // ranks, 1-based, one per level
};

// (depth, then lexicographic) order of rank paths
bool path_less(const std::vector<int> &a, const std::vector<int> &b) {
    if (a.size() != b.size()) return a.size() < b.size();
    return a < b;
}

// heap order: the top is the largest product, then the smaller depth, then the smaller path
struct Worse {
    bool operator()(const Cand &x, const Cand &y) const {
        if (x.v != y.v) return x.v < y.v;
        return path_less(y.path, x.path);
    }
};

constexpr int kMaxTreeNodes = 16384;  // the tree mask's limit
constexpr int kMaxHeads = 64;
constexpr int kMaxRanks = 4096;

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" spec_status spec_build_sparse_tree(const double *accuracy, int K, int S, int n_nodes, int32_t *parents,
                                              int32_t *depth, int32_t *rank, int *n_built, double *expected_len) {
    if (K < 1 || K > kMaxHeads || S < 1 || S > kMaxRanks || n_nodes < 1 || n_nodes > kMaxTreeNodes)
        return fail(SPEC_ERR_INVALID_ARG, "need 1 <= K <= %d, 1 <= S <= %d, 1 <= n_nodes <= %d (K=%d S=%d n=%d)",
                    kMaxHeads, kMaxRanks, kMaxTreeNodes, K, S, n_nodes);
    if (!accuracy || !parents || !depth || !rank || !n_built) return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    for (int q = 0; q < K * S; ++q)
        if (!(accuracy[q] >= 0.0 && accuracy[q] <= 1.0))
            return fail(SPEC_ERR_INVALID_ARG, "accuracy[%d] = %g is not in [0, 1]", q, accuracy[q]);
    std::vector<Cand> chosen;
    chosen.reserve(static_cast<size_t>(n_nodes));
    chosen.push_back(Cand{1.0, {}});  // the root
    std::priority_queue<Cand, std::vector<Cand>, Worse> heap;
    auto push_children = [&](const Cand &p) {
        const size_t m = p.path.size();
        if (m >= static_cast<size_t>(K)) return;
        for (int i = 1; i <= S; ++i) {
            Cand c{p.v * accuracy[m * static_cast<size_t>(S) + (i - 1)], p.path};
            c.path.push_back(i);
            heap.push(std::move(c));
        }
    };
    push_children(chosen[0]);
    while (static_cast<int>(chosen.size()) < n_nodes && !heap.empty()) {
        chosen.push_back(heap.top());
        heap.pop();
        push_children(chosen.back());
    }
    // number by (depth, rank path); parents through a map from path to number
    std::vector<int> order(chosen.size());
    for (size_t q = 0; q < order.size(); ++q) order[q] = static_cast<int>(q);
    std::sort(order.begin(), order.end(),
              [&](int a, int b) { return path_less(chosen[a].path, chosen[b].path); });
    std::map<std::vector<int>, int> number;
    double e = 0.0;
    for (size_t r = 0; r < order.size(); ++r) {
        const Cand &c = chosen[order[r]];
        number[c.path] = static_cast<int>(r);
        const size_t m = c.path.size();
        depth[r] = static_cast<int32_t>(m);
        rank[r] = m ? c.path.back() : 0;
        parents[r] = -1;
        if (m) {
            parents[r] = number.at(std::vector<int>(c.path.begin(), c.path.end() - 1));
            e += c.v;
        }
    }
    *n_built = static_cast<int>(order.size());
    if (expected_len) *expected_len = e;
    return SPEC_OK;
}
