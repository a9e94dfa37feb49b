// peer_select.cu -- SAPS bandwidth-aware peer selection (host code only).
//
// Source: "Communication-Efficient Decentralized Learning with Sparsification
// and Adaptive Peer Selection", section II-C (gossip matrix generation,
// Algorithm 3) and section II-A (the coordinator filters the bandwidth matrix
// B with B_thres into B*).
//
// One round:
//   1. B is symmetrised with the slower direction, B_ij = B_ji = min(B_ij, B_ji).
//   2. B*: the pairs whose bandwidth exceeds B_thres.
//   3. The "recently connected" (RC) edges are the pairs (i, j) last matched
//      in a round r with r > t - T_thres.  If they connect all workers, the
//      candidate graph E is B*; otherwise E holds the links of B (B_ij > 0)
//      between different connected components of the RC graph, so that the
//      round joins components.
//   4. A maximum matching of E (Edmonds' blossom algorithm for general
//      graphs), started from a seeded random relabelling of the workers.
//   5. The workers left unmatched are paired among themselves in a seeded
//      random order, without regard to bandwidth.
//   6. The pairs are the round's perfect matching (its gossip matrix puts 1/2
//      on i,i / i,j / j,i / j,j for each pair: doubly stochastic), and R_ij,
//      R_ji are set to t for each pair.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "gc_common.cuh"
#include "../../include/gc_gb300_testing.h"

namespace gc {
namespace {

// Fisher-Yates permutation of 0..n-1 from a seed: the swap partner of
// position i (counting down) is splitmix64(key ^ i) mod (i + 1).
void seeded_permutation(uint64_t key, int n, int* perm) {
    for (int i = 0; i < n; ++i) perm[i] = i;
    for (int i = n - 1; i > 0; --i) {
        const int j = static_cast<int>(splitmix64(key ^ static_cast<uint64_t>(i)) % static_cast<uint64_t>(i + 1));
        std::swap(perm[i], perm[j]);
    }
}

// Connected components of an undirected graph given as an n x n 0/1 matrix;
// comp[v] = smallest vertex of v's component.  Returns the component count.
int components(int n, const std::vector<uint8_t>& adj, std::vector<int>& comp) {
    comp.assign(n, -1);
    int count = 0;
    std::vector<int> stack;
    for (int s = 0; s < n; ++s) {
        if (comp[s] >= 0) continue;
        ++count;
        comp[s] = s;
        stack.assign(1, s);
        while (!stack.empty()) {
            const int v = stack.back();
            stack.pop_back();
            for (int u = 0; u < n; ++u)
                if (adj[v * n + u] && comp[u] < 0) {
                    comp[u] = s;
                    stack.push_back(u);
                }
        }
    }
    return count;
}

// Maximum-cardinality matching of a general graph (Edmonds 1965): grow an
// alternating tree from each free vertex by breadth-first search; an edge
// between two outer vertices of the tree closes an odd cycle, which is
// shrunk into its base (every vertex of the cycle becomes outer); reaching a
// free vertex gives an augmenting path, which flips the matching along it.
class BlossomMatcher {
public:
    BlossomMatcher(int n, const std::vector<uint8_t>& adj) : n_(n), adj_(adj), mate_(n, -1) {}

    const std::vector<int>& run() {
        for (int root = 0; root < n_; ++root)
            if (mate_[root] < 0) grow_from(root);
        return mate_;
    }

private:
    int n_;
    const std::vector<uint8_t>& adj_;
    std::vector<int> mate_;
    std::vector<int> parent_;     // tree edge into an inner vertex
    std::vector<int> base_;       // base of the shrunk blossom holding v
    std::vector<uint8_t> outer_;  // v is an outer (even) vertex of the tree
    std::vector<int> queue_;

    // The base of the lowest common blossom of outer vertices a and b.
    int common_base(int a, int b) const {
        std::vector<uint8_t> seen(n_, 0);
        for (;;) {
            a = base_[a];
            seen[a] = 1;
            if (mate_[a] < 0) break;          // reached the root
            a = parent_[mate_[a]];
        }
        for (;;) {
            b = base_[b];
            if (seen[b]) return b;
            b = parent_[mate_[b]];
        }
    }

    // Marks the blossoms on the tree path from v up to base `b`, and points
    // the inner vertices on it back across the closing edge (towards `child`).
    void mark_path(int v, int b, int child, std::vector<uint8_t>& in_cycle) {
        while (base_[v] != b) {
            in_cycle[base_[v]] = in_cycle[base_[mate_[v]]] = 1;
            parent_[v] = child;
            child = mate_[v];
            v = parent_[mate_[v]];
        }
    }

    void shrink(int v, int u) {
        const int b = common_base(v, u);
        std::vector<uint8_t> in_cycle(n_, 0);
        mark_path(v, b, u, in_cycle);
        mark_path(u, b, v, in_cycle);
        for (int x = 0; x < n_; ++x)
            if (in_cycle[base_[x]]) {
                base_[x] = b;
                if (!outer_[x]) {
                    outer_[x] = 1;
                    queue_.push_back(x);
                }
            }
    }

    void augment(int v) {
        while (v >= 0) {
            const int p = parent_[v];
            const int next = mate_[p];
            mate_[v] = p;
            mate_[p] = v;
            v = next;
        }
    }

    void grow_from(int root) {
        parent_.assign(n_, -1);
        outer_.assign(n_, 0);
        base_.resize(n_);
        for (int v = 0; v < n_; ++v) base_[v] = v;
        queue_.assign(1, root);
        outer_[root] = 1;
        for (size_t head = 0; head < queue_.size(); ++head) {
            const int v = queue_[head];
            for (int u = 0; u < n_; ++u) {
                if (!adj_[v * n_ + u] || base_[v] == base_[u] || mate_[v] == u) continue;
                if (u == root || (mate_[u] >= 0 && parent_[mate_[u]] >= 0)) {
                    shrink(v, u);                 // u is outer: an odd cycle
                } else if (parent_[u] < 0) {
                    parent_[u] = v;               // u becomes inner
                    if (mate_[u] < 0) {
                        augment(u);
                        return;
                    }
                    outer_[mate_[u]] = 1;
                    queue_.push_back(mate_[u]);
                }
            }
        }
    }
};

}  // namespace
}  // namespace gc

using namespace gc;

extern "C" int saps_matching_bandwidth(int W, const double* bandwidth, double b_thres, int64_t* last_round,
                                       int64_t t, int64_t t_thres, uint64_t seed_t, int* pairs_out) {
    if (W < 2 || W > GC_MAX_WORKERS || (W & 1) || !bandwidth || !last_round || !pairs_out || t_thres < 1)
        return GC_ERR_INVALID;
    if (!(b_thres == b_thres)) return GC_ERR_INVALID;
    for (int i = 0; i < W * W; ++i)
        if (!(bandwidth[i] >= 0.0) || bandwidth[i] == INFINITY) return GC_ERR_INVALID;
    // 1-3: symmetrised bandwidth, its filtered graph, the RC graph
    std::vector<double> B(W * W, 0.0);
    std::vector<uint8_t> rc(W * W, 0), cand(W * W, 0);
    for (int i = 0; i < W; ++i)
        for (int j = 0; j < W; ++j)
            if (i != j) {
                B[i * W + j] = std::min(bandwidth[i * W + j], bandwidth[j * W + i]);
                const int64_t r = std::max(last_round[i * W + j], last_round[j * W + i]);
                rc[i * W + j] = r > t - t_thres;
            }
    std::vector<int> comp;
    if (components(W, rc, comp) == 1) {
        for (int i = 0; i < W * W; ++i) cand[i] = B[i] > b_thres;
    } else {
        for (int i = 0; i < W; ++i)
            for (int j = 0; j < W; ++j)
                cand[i * W + j] = i != j && comp[i] != comp[j] && B[i * W + j] > 0.0;
    }
    // 4: maximum matching of the candidate graph on a seeded relabelling
    std::vector<int> perm(W), label_of(W);
    seeded_permutation(splitmix64(seed_t ^ 0x243F6A8885A308D3ull), W, perm.data());
    for (int k = 0; k < W; ++k) label_of[perm[k]] = k;      // worker perm[k] is vertex k
    std::vector<uint8_t> adj(W * W, 0);
    for (int i = 0; i < W; ++i)
        for (int j = 0; j < W; ++j) adj[label_of[i] * W + label_of[j]] = cand[i * W + j];
    BlossomMatcher matcher(W, adj);
    const std::vector<int>& mate_lab = matcher.run();
    std::vector<int> mate(W, -1);
    for (int k = 0; k < W; ++k)
        if (mate_lab[k] >= 0) mate[perm[k]] = perm[mate_lab[k]];
    // 5: the unmatched workers, paired in a seeded random order
    std::vector<int> free_w;
    for (int i = 0; i < W; ++i)
        if (mate[i] < 0) free_w.push_back(i);
    if (!free_w.empty()) {
        const int m = static_cast<int>(free_w.size());
        std::vector<int> fp(m);
        seeded_permutation(splitmix64(seed_t ^ 0x13198A2E03707344ull), m, fp.data());
        for (int q = 0; q + 1 < m; q += 2) {
            const int a = free_w[fp[q]], b = free_w[fp[q + 1]];
            mate[a] = b;
            mate[b] = a;
        }
    }
    // 6: pairs (smaller worker first, pairs in order of their first worker),
    // and the round stamps
    int k = 0;
    for (int i = 0; i < W; ++i) {
        if (mate[i] < 0 || mate[mate[i]] != i) return GC_ERR_INVALID;   // cannot happen for even W
        if (mate[i] > i) {
            pairs_out[k++] = i;
            pairs_out[k++] = mate[i];
            last_round[i * W + mate[i]] = t;
            last_round[mate[i] * W + i] = t;
        }
    }
    return GC_OK;
}

// The Elias decoders' CTA sizing rule, on given sizes (no device needed).
extern "C" int gc_testing_decode_buckets_per_cta(int64_t nb, int W, int64_t slots, int maxb, int64_t* bpc) {
    if (nb < 1 || nb > (int64_t{1} << 40) || W < 1 || W > GC_MAX_WORKERS || slots < 1 ||
        slots > (int64_t{1} << 20) || maxb < 1 || maxb > 1024 || !bpc)
        return GC_ERR_INVALID;
    *bpc = gc::even_buckets_per_cta(nb, W, slots, maxb);
    return GC_OK;
}

// The CUDA runtime's L2 fetch-granularity hint of the current context (a
// per-process limit); see the header.  Random 4-byte gathers move less DRAM
// traffic per value at 32 or 64 bytes than at 128.
extern "C" int gc_l2_fetch_granularity(size_t bytes, size_t* previous) {
    if (bytes > 128) return GC_ERR_INVALID;
    size_t old = 0;
    if (cudaDeviceGetLimit(&old, cudaLimitMaxL2FetchGranularity) != cudaSuccess) return GC_ERR_CUDA;
    if (cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, bytes) != cudaSuccess) return GC_ERR_CUDA;
    if (previous) *previous = old;
    return GC_OK;
}
