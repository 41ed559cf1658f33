"""Pins of the oracle's dynamic draft tree against what the algorithm fixes: a top-1 tree is
the greedy chain with its closed-form confidences; on tiny vocabularies the nodes are
exactly the highest-confidence members of the complete (depth-limited, top-k) candidate
tree, enumerated by brute force; confidences are products along the path; the threshold
and the depth limit hold; ties go to the lower token id and to the earlier candidate."""

import numpy as np
import pytest

import oracle.draft_tree as DT


def _rows(seed, n, V, scale=2.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, V)) * scale).astype(np.float32)


def _softmax(x):
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def test_topk_softmax_matches_sort_and_ties_to_lower_id():
    row = np.array([1.0, 3.0, 3.0, -2.0, 3.0, 0.5], np.float32)
    idx, p = DT.topk_softmax(row, 4)
    assert idx.tolist() == [1, 2, 4, 0]
    np.testing.assert_allclose(p, _softmax(row)[[1, 2, 4, 0]], rtol=1e-15)


def test_top1_tree_is_the_greedy_chain():
    V, n, depth = 11, 6, 8
    rows = _rows(1, n, V)
    parent, token, score, tight = DT.best_first_tree(lambda u: rows[u], 7, n, 1, depth)
    assert parent.tolist() == [-1, 0, 1, 2, 3, 4]
    want_tok = [7] + [int(np.argmax(rows[u])) for u in range(n - 1)]
    assert token.tolist() == want_tok
    want = np.cumprod([1.0] + [_softmax(rows[u]).max() for u in range(n - 1)])
    np.testing.assert_allclose(score, want, rtol=1e-14)
    assert not tight


def test_depth_limit_stops_the_chain():
    rows = _rows(2, 10, 9)
    parent, token, score, _ = DT.best_first_tree(lambda u: rows[u], 0, 10, 1, 3)
    assert parent.tolist() == [-1, 0, 1, 2]   # depth 3 reached, nothing else queued


def _complete_tree(row_of_path, V, k, max_depth):
    """Every node of the complete candidate tree (token paths of length 1..max_depth, each
    step among the parent's top-k): (path tuple, confidence)."""
    out = []
    frontier = [((), 1.0)]
    for _ in range(max_depth):
        nxt = []
        for path, c in frontier:
            p = _softmax(row_of_path(path))
            top = np.lexsort((np.arange(V), -np.asarray(row_of_path(path), np.float64)))[:k]
            for t in top:
                node = (path + (int(t),), c * p[t])
                out.append(node)
                nxt.append(node)
        frontier = nxt
    return out


@pytest.mark.parametrize("seed,V,k,depth,n", [(3, 5, 2, 3, 6), (4, 6, 3, 2, 8), (5, 4, 2, 4, 9), (6, 7, 3, 3, 12)])
def test_nodes_are_the_top_confidences_of_the_complete_tree(seed, V, k, depth, n):
    """Confidences fall along every path, so the best-first nodes are exactly the n - 1
    highest-confidence members of the complete candidate tree, in falling order. The
    expected node ids come from a global sort of that tree (brute force, no queue); the
    oracle is driven with rows looked up by those ids, so a different pop order shows up as
    a token that does not extend its parent's path."""
    rng = np.random.default_rng(seed)
    table = {}

    def row_of_path(path):   # one fixed logits row per token path (what the draft model sees)
        if path not in table:
            table[path] = (rng.standard_normal(V) * 2.0).astype(np.float32)
        return table[path]

    full = _complete_tree(row_of_path, V, k, depth)
    ranked = sorted(full, key=lambda node: -node[1])
    id_path = [()] + [path for path, _ in ranked[: n - 1]]
    parent, token, score, tight = DT.best_first_tree(lambda u: row_of_path(id_path[u]), 0, n, k, depth)
    assert len(parent) == n
    for u in range(1, n):
        assert parent[u] < u
        p_path = id_path[parent[u]]
        assert id_path[u] == p_path + (int(token[u]),)
        np.testing.assert_allclose(score[u], score[parent[u]] * _softmax(row_of_path(p_path))[token[u]],
                                   rtol=1e-13)
        np.testing.assert_allclose(score[u], ranked[u - 1][1], rtol=1e-13)
    assert np.all(np.diff(score[1:]) <= 0)   # nodes leave the queue in falling confidence


def test_threshold_drops_candidates():
    rows = _rows(7, 20, 6, scale=1.0)
    parent, token, score, _ = DT.best_first_tree(lambda u: rows[u], 0, 20, 3, 5, threshold=0.05)
    assert (score[1:] > 0.05).all()
    parent2, token2, score2, _ = DT.best_first_tree(lambda u: rows[u], 0, 20, 3, 5)
    assert len(parent2) == 20 and (score2[1:] <= 0.05).any()


def test_ties_go_to_the_earlier_candidate():
    # a uniform row: the root's top-2 children tie; the first queued (lower token) is node 1
    rows = np.zeros((4, 4), np.float32)
    parent, token, score, tight = DT.best_first_tree(lambda u: rows[u], 0, 4, 2, 1)
    assert token.tolist() == [0, 0, 1] and parent.tolist() == [-1, 0, 0]
    assert tight


def test_edge_keyed_rows_reach_the_node_they_define():
    """row_key="edge" hands row_of the node's own parent and token: the same tree comes out
    when the rows are looked up by node id from the finished tree."""
    from draft_protocol import EdgeRows
    er = EdgeRows(3, 50, scale=1.5)
    parent, token, score, _ = DT.best_first_tree(er.of(0), 5, 24, 4, 4, row_key="edge")
    by_node = [er.row(0, parent[u], token[u]) for u in range(len(parent))]
    parent2, token2, score2, _ = DT.best_first_tree(lambda u: by_node[u], 5, 24, 4, 4)
    assert np.array_equal(parent, parent2) and np.array_equal(token, token2)
    np.testing.assert_array_equal(score, score2)


@pytest.mark.parametrize("seed,V,k,depth,n,thr,bump", [
    (1, 64, 10, 8, 64, 0.0, 0.0), (2, 40, 4, 6, 48, 0.0, 0.0), (3, 30, 16, 3, 100, 0.0, 0.0),
    (4, 25, 1, 8, 9, 0.0, 0.0), (5, 100, 3, 5, 32, 0.05, 0.0), (6, 64, 10, 8, 64, 0.0, 6.0),
    (7, 16, 2, 12, 80, 0.0, 3.0)])
def test_multi_row_protocol_builds_the_pages_tree(seed, V, k, depth, n, thr, bump):
    """The batched protocol (several rows per call, results kept per candidate, pops replayed)
    gives the one-pop-at-a-time tree for every width; width 1 takes one call per expanded
    node; a wider call never needs more calls; every request is a distinct (parent, token)."""
    from draft_protocol import EdgeRows, multi_row_tree
    er = EdgeRows(seed, V, scale=2.0, bump=bump)
    want_p, want_t, _, _ = DT.best_first_tree(er.of(0), 1, n, k, depth, threshold=thr, row_key="edge")
    calls = {}
    for w in (1, 2, 3, 8):
        run = multi_row_tree(er.of(0), 1, n, k, depth, w, threshold=thr)
        assert np.array_equal(run.parent, want_p) and np.array_equal(run.token, want_t), w
        seen = [rq for call in run.requests for rq in call]
        assert len(seen) == len(set(seen)), "a row was requested twice"
        assert all(len(call) <= w for call in run.requests)
        calls[w] = run.calls
    d = [0] * len(want_p)
    for u in range(1, len(want_p)):
        d[u] = d[want_p[u]] + 1
    expanded = sum(1 for u in range(len(want_p)) if d[u] < depth and u < n - 1)   # nodes that needed a row
    assert calls[1] == expanded
    assert calls[8] <= calls[3] <= calls[1] and calls[2] <= calls[1]
