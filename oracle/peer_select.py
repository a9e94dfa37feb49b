"""Oracle for SAPS bandwidth-aware peer selection (test infrastructure).

Only ``tests/`` may import this module; the product library never does.

Source: "Communication-Efficient Decentralized Learning with Sparsification
and Adaptive Peer Selection", section II-A (the coordinator filters the
bandwidth matrix B with B_thres into B*) and section II-C (Algorithm 3:
symmetrised bandwidth, "recently connected" edges, the connectivity test,
edges that join the RC components, maximum matching, then the unmatched
workers paired without regard to bandwidth).

The matching itself is randomised on the page (RandomlyMaxMatch), so the
oracle gives what is unique about a round: the candidate graph E and the size
of a maximum matching of E, found by exhaustive search (small W only).  A
correct round's perfect matching uses exactly that many E edges.
"""
from __future__ import annotations

from functools import lru_cache

import numpy as np


def symmetrise(B: np.ndarray) -> np.ndarray:
    """B_ij = B_ji = min(B_ij, B_ji): a link is as fast as its slower direction."""
    B = np.asarray(B, dtype=np.float64)
    S = np.minimum(B, B.T)
    np.fill_diagonal(S, 0.0)
    return S


def rc_components(last_round: np.ndarray, t: int, t_thres: int) -> list[int]:
    """Label of each worker's connected component in the graph of recently
    connected pairs (last matched in a round r with r > t - t_thres); the
    label is the smallest worker of the component."""
    W = last_round.shape[0]
    rc = np.maximum(last_round, last_round.T) > t - t_thres
    label = list(range(W))
    changed = True
    while changed:                      # propagate the smallest label along RC edges
        changed = False
        for i in range(W):
            for j in range(W):
                if i != j and rc[i, j] and label[j] < label[i]:
                    label[i] = label[j]
                    changed = True
    return label


def candidate_graph(B: np.ndarray, b_thres: float, last_round: np.ndarray, t: int, t_thres: int):
    """(E, connected): the pairs the round's maximum matching may use.  If the
    RC graph connects every worker, E is B* (pairs faster than b_thres);
    otherwise E is every link (B_ij > 0) between two different RC components."""
    S = symmetrise(B)
    label = rc_components(last_round, t, t_thres)
    W = S.shape[0]
    connected = len(set(label)) == 1
    E = np.zeros((W, W), dtype=bool)
    for i in range(W):
        for j in range(W):
            if i == j:
                continue
            E[i, j] = S[i, j] > b_thres if connected else (label[i] != label[j] and S[i, j] > 0.0)
    return E, connected


def max_matching_size(E: np.ndarray) -> int:
    """Size of a maximum matching of the graph E by exhaustive search: the
    lowest unmatched vertex is either left out or matched to each neighbour."""
    W = E.shape[0]
    adj = [frozenset(int(j) for j in np.nonzero(E[i])[0]) for i in range(W)]

    @lru_cache(maxsize=None)
    def best(free: frozenset) -> int:
        if len(free) < 2:
            return 0
        v = min(free)
        rest = free - {v}
        out = best(rest)
        for u in adj[v] & rest:
            out = max(out, 1 + best(rest - {u}))
        return out

    return best(frozenset(range(W)))
