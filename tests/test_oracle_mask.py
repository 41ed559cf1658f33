"""Pins of the oracle's ancestor mask against what the pages and the mathematics fix.

Definition pinned: "EAGLE-2 deep dive", core-implementation section — a node's
mask row marks the node and each ancestor up to the root.
"""

import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _subtree_sets(parent):
    """Brute force from the other direction: for every node j, the set of nodes
    in j's subtree, by breadth-first search down the child lists."""
    n = len(parent)
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[parent[i]].append(i)
    out = []
    for j in range(n):
        seen, frontier = {j}, [j]
        while frontier:
            nxt = []
            for v in frontier:
                for c in kids[v]:
                    seen.add(c)
                    nxt.append(c)
            frontier = nxt
        out.append(seen)
    return out


def _random_parent(rng, n, max_depth=None):
    parent = [-1]
    depth = [0]
    for i in range(1, n):
        cands = [j for j in range(i) if max_depth is None or depth[j] < max_depth]
        p = int(rng.choice(cands))
        parent.append(p)
        depth.append(depth[p] + 1)
    return np.asarray(parent)


def test_golden_small_tree():
    g = json.load(open(os.path.join(GOLDEN, "tree_mask_small.json")))
    M, depth = oracle.ancestor_mask(g["parent"])
    n = len(g["parent"])
    want = np.zeros((n, n), bool)
    for i, row in enumerate(g["mask_rows"]):
        want[i, row] = True
    assert np.array_equal(M, want)
    assert depth.tolist() == g["depth"]
    words = oracle.pack_mask_words(M, 1)[:, 0]
    assert [hex(int(w)) for w in words] == g["mask_words_hex"]


@pytest.mark.parametrize("seed", range(20))
def test_mask_equals_bruteforce_subtrees(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 70))
    parent = _random_parent(rng, n, max_depth=None if seed % 2 else 8)
    M, depth = oracle.ancestor_mask(parent)
    sub = _subtree_sets(parent)
    want = np.array([[i in sub[j] for j in range(n)] for i in range(n)])
    assert np.array_equal(M, want)
    # invariants: self bit, root bit, lower triangular, popcount = depth + 1
    assert M[np.arange(n), np.arange(n)].all()
    assert M[:, 0].all()
    assert not np.triu(M, 1).any()
    assert np.array_equal(M.sum(1), depth + 1)
    # depth = number of hops to the root, counted independently
    for i in range(n):
        hops, v = 0, i
        while parent[v] >= 0:
            v, hops = parent[v], hops + 1
        assert depth[i] == hops


def test_chain_is_lower_triangular_ones():
    n = 9
    M, depth = oracle.ancestor_mask(np.arange(-1, n - 1))
    assert np.array_equal(M, np.tril(np.ones((n, n), bool)))
    assert depth.tolist() == list(range(n))


def test_star_tree():
    n = 12
    M, depth = oracle.ancestor_mask([-1] + [0] * (n - 1))
    want = np.eye(n, dtype=bool)
    want[:, 0] = True
    assert np.array_equal(M, want)


@pytest.mark.parametrize("bad", [[0, 0], [-1, 1], [-1, 0, 3], [-1, -1], [-1, 0, 2]])
def test_rejects_invalid_parent(bad):
    with pytest.raises(ValueError):
        oracle.ancestor_mask(bad)


def test_batch_layout_and_words():
    rng = np.random.default_rng(7)
    parents = [_random_parent(rng, n) for n in (5, 1, 130, 64)]
    qo = np.concatenate([[0], np.cumsum([len(p) for p in parents])])
    mask, depth = oracle.ancestor_mask_batch(np.concatenate(parents), qo)
    assert mask.shape == (qo[-1], 130)
    words = oracle.pack_mask_words(mask, 3)
    for b, p in enumerate(parents):
        M, d = oracle.ancestor_mask(p)
        a = qo[b]
        assert np.array_equal(mask[a : a + len(p), : len(p)], M)
        assert not mask[a : a + len(p), len(p):].any()
        for i in range(len(p)):
            for j in range(len(p)):
                bit = (int(words[a + i, j >> 6]) >> (j & 63)) & 1
                assert bit == int(M[i, j])
