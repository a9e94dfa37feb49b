"""SAPS bandwidth-aware peer selection (Algorithm 3 of "Communication-Efficient
Decentralized Learning with Sparsification and Adaptive Peer Selection",
section II-C), host code: the oracle's pins, then the library function
``saps_matching_bandwidth`` against the oracle.

The page's matching is randomised, so what is compared is what every correct
round shares: the result is a perfect matching, exactly nu(E) of its pairs are
candidate pairs (nu(E) = size of a maximum matching of the candidate graph E,
found by exhaustive search), the round stamps move to t for the chosen pairs
only, and the gossip matrix is doubly stochastic.
"""
import ctypes

import numpy as np
import pytest

import gradient_compression_sgd_gc_gb300 as gc
from oracle import peer_select as ps

NEVER = gc.NEVER


def _graph(W, edges):
    E = np.zeros((W, W), dtype=bool)
    for a, b in edges:
        E[a, b] = E[b, a] = True
    return E


# ---------------------------------------------------------------- oracle pins

@pytest.mark.parametrize("W,edges,nu", [
    (6, [(i, i + 1) for i in range(5)], 3),                              # path P6
    (7, [(i, i + 1) for i in range(6)], 3),                              # path P7
    (5, [(i, (i + 1) % 5) for i in range(5)], 2),                        # odd cycle C5
    (6, [(i, (i + 1) % 6) for i in range(6)], 3),                        # even cycle C6
    (6, [(0, k) for k in range(1, 6)], 1),                               # star K1,5
    (7, [(a, b) for a in range(7) for b in range(a + 1, 7)], 3),         # complete K7
    (6, [(0, 1), (1, 2), (2, 0), (3, 4), (4, 5), (5, 3)], 2),            # two triangles
    (5, [(0, 1), (1, 2), (2, 0), (2, 3), (3, 4), (4, 2)], 2),            # bowtie
    (4, [], 0),
    # Petersen graph: outer 5-cycle, inner pentagram, spokes (perfect matching of 5)
    (10, [(i, (i + 1) % 5) for i in range(5)] + [(5 + i, 5 + (i + 2) % 5) for i in range(5)]
     + [(i, i + 5) for i in range(5)], 5),
    # a blossom hides the augmenting path: triangle 1-2-3 with tails 0-1 and 3-4, 2-5
    (6, [(0, 1), (1, 2), (2, 3), (3, 1), (3, 4), (2, 5)], 3),
])
def test_max_matching_size_closed_forms(W, edges, nu):
    assert ps.max_matching_size(_graph(W, edges)) == nu


def test_symmetrise_takes_the_slower_direction():
    B = np.array([[7, 3, 5], [4, 0, 9], [1, 2, 8]], dtype=float)
    np.testing.assert_array_equal(ps.symmetrise(B), [[0, 3, 1], [3, 0, 2], [1, 2, 0]])


def test_rc_components_and_candidate_graph_by_hand():
    W = 4
    B = np.array([[0, 9, 1, 9], [9, 0, 9, 1], [1, 9, 0, 9], [9, 1, 9, 0]], dtype=float)
    R = np.full((W, W), NEVER, np.int64)
    R[0, 1] = R[1, 0] = 10                       # recent (t = 11, t_thres = 3)
    R[2, 3] = R[3, 2] = 7                        # too old: 7 <= 11 - 3
    assert ps.rc_components(R, 11, 3) == [0, 0, 2, 3]
    E, connected = ps.candidate_graph(B, 5.0, R, 11, 3)
    assert not connected
    # links between different components, whatever their bandwidth
    assert not E[0, 1] and E[0, 2] and E[0, 3] and E[1, 2] and E[1, 3] and E[2, 3]
    R[1, 2] = R[2, 1] = R[2, 3] = R[3, 2] = 10
    E, connected = ps.candidate_graph(B, 5.0, R, 11, 3)
    assert connected
    np.testing.assert_array_equal(E, ps.symmetrise(B) > 5.0)     # B* once connected


# ---------------------------------------------------------------- the library function

def _check_round(W, B, b_thres, R, t, t_thres, seed):
    R0 = R.copy()
    E, connected = ps.candidate_graph(B, b_thres, R0, t, t_thres)
    pairs = gc.saps_matching_bandwidth(B, b_thres, R, t, t_thres, seed)
    assert sorted(pairs) == list(range(W)), "not a perfect matching"
    pl = [(pairs[q], pairs[q + 1]) for q in range(0, W, 2)]
    assert all(a < b for a, b in pl) and [a for a, _ in pl] == sorted(a for a, _ in pl)
    assert sum(bool(E[a, b]) for a, b in pl) == ps.max_matching_size(E)
    expect = R0.copy()
    for a, b in pl:
        expect[a, b] = expect[b, a] = t
    np.testing.assert_array_equal(R, expect)
    M = gc.gossip_matrix(pairs)
    np.testing.assert_array_equal(M.sum(0), np.ones(W))
    np.testing.assert_array_equal(M.sum(1), np.ones(W))
    np.testing.assert_array_equal(M, M.T)
    return pl, E, connected


@pytest.mark.parametrize("W", [2, 4, 6, 8, 10])
def test_rounds_against_oracle(W):
    rng = np.random.default_rng(100 + W)
    for case in range(40):
        B = rng.uniform(0.5, 10.0, (W, W))
        B[rng.random((W, W)) < 0.2] = 0.0                      # some missing links
        b_thres = float(rng.uniform(2.0, 8.0))
        t_thres = int(rng.integers(1, 6))
        R = np.full((W, W), NEVER, np.int64)
        for t in range(8):                                      # consecutive rounds share R
            _check_round(W, B, b_thres, R, t, t_thres, gc.saps_round_seed(case, t))


def test_first_round_bridges_every_worker_and_later_rounds_use_fast_links():
    """Round 0 has no recent edges, so every worker is its own component and
    every link is a candidate; the RC graph then gains a perfect matching per
    round, and once it connects all 16 workers (after at most log2 16 rounds
    with a long T_thres) only links faster than b_thres are candidates."""
    W, t_thres = 16, 1000
    rng = np.random.default_rng(3)
    B = rng.uniform(1.0, 10.0, (W, W))
    R = np.full((W, W), NEVER, np.int64)
    connected_at = None
    for t in range(10):
        pl, E, connected = _check_round(W, B, 4.0, R, t, t_thres, gc.saps_round_seed(9, t))
        if connected and connected_at is None:
            connected_at = t
        if not connected:
            comp = ps.rc_components(R, t, t_thres)
            assert len(set(comp)) <= max(1, W >> (t + 1))      # components at least halve
        else:
            fast = ps.symmetrise(B) > 4.0
            if ps.max_matching_size(fast) == W // 2:
                assert all(fast[a, b] for a, b in pl)
    assert connected_at is not None and connected_at <= 4


def test_deterministic_and_seed_dependent():
    W = 12
    rng = np.random.default_rng(8)
    B = rng.uniform(1.0, 10.0, (W, W))
    outs = set()
    for seed in range(20):
        R1 = np.full((W, W), NEVER, np.int64)
        R2 = R1.copy()
        p1 = gc.saps_matching_bandwidth(B, 3.0, R1, 0, 5, seed)
        p2 = gc.saps_matching_bandwidth(B, 3.0, R2, 0, 5, seed)
        assert p1 == p2
        outs.add(tuple(p1))
    assert len(outs) > 10


@pytest.mark.parametrize("W", [16, 64])
def test_large_rounds_against_networkx(W):
    nx = pytest.importorskip("networkx")
    rng = np.random.default_rng(W)
    for case in range(10):
        B = rng.uniform(0.0, 10.0, (W, W))
        R = np.full((W, W), NEVER, np.int64)
        for t in range(7):
            R0 = R.copy()
            E, _ = ps.candidate_graph(B, 6.0, R0, t, 3)
            pairs = gc.saps_matching_bandwidth(B, 6.0, R, t, 3, gc.saps_round_seed(case, t))
            assert sorted(pairs) == list(range(W))
            G = nx.Graph()
            G.add_nodes_from(range(W))
            G.add_edges_from((i, j) for i in range(W) for j in range(i + 1, W) if E[i, j])
            nu = len(nx.max_weight_matching(G, maxcardinality=True))
            assert sum(bool(E[pairs[q], pairs[q + 1]]) for q in range(0, W, 2)) == nu


def test_validation():
    lib = gc.load()
    W = 4
    B = np.ones((W, W))
    R = np.full((W, W), NEVER, np.int64)
    out = (ctypes.c_int * 8)()

    def call(W=4, B=B, thr=1.0, R=R, t=0, tt=3):
        return lib.saps_matching_bandwidth(W, B.ctypes.data, thr, R.ctypes.data, t, tt, 1, out)
    assert call() == gc.GC_OK
    assert call(W=3) == gc.GC_ERR_INVALID
    assert call(W=0) == gc.GC_ERR_INVALID
    assert call(W=66) == gc.GC_ERR_INVALID
    assert call(thr=float("nan")) == gc.GC_ERR_INVALID
    assert call(tt=0) == gc.GC_ERR_INVALID
    bad = B.copy()
    bad[1, 2] = -1.0
    assert call(B=bad) == gc.GC_ERR_INVALID
    bad[1, 2] = float("inf")
    assert call(B=bad) == gc.GC_ERR_INVALID
    assert lib.saps_matching_bandwidth(4, None, 1.0, R.ctypes.data, 0, 3, 1, out) == gc.GC_ERR_INVALID
    with pytest.raises(ValueError):
        gc.saps_matching_bandwidth(B, 1.0, R.astype(np.int32), 0, 3, 1)
