"""CPU check of the bench's accept-depth workloads: plant_accept_depth changes the target
logits so that greedy acceptance (the oracle's) takes exactly d nodes along lowest-id
children in every sequence whose tree reaches depth d, for the single-sequence workload and a
small batch of EAGLE-2 trees; rows off the planted path are left as they were."""

import numpy as np

import bench
import oracle
from speculative_decoding_tree_parent_gb300 import workloads as W


def _first_child_path(par, a, e, d):
    path, v = [0], 0
    for _ in range(d):
        kids = [c for c in range(v + 1, e - a) if par[a + c] == v]
        if not kids:
            break
        v = kids[0]
        path.append(v)
    return path


def test_plant_accept_depth_single_sequence():
    inp = W.generate_index(2)
    for d in range(inp.path_cap):
        tl = bench.plant_accept_depth(inp, d)
        ref = oracle.greedy_accept(inp.parent, inp.draft_tokens, tl, inp.qo_indptr, inp.path_cap)
        assert ref.accept_len.tolist() == [d]
        want = _first_child_path(np.asarray(inp.parent), 0, int(inp.qo_indptr[1]), d)
        assert ref.path[0, : d + 1].tolist() == want
        off = np.setdiff1d(np.arange(tl.shape[0]), want)
        assert np.array_equal(tl[off], inp.target_logits[off])


def test_plant_accept_depth_batch():
    inp = W.generate(W.spec(3, batch=6, nodes=(24, 24), vocab=512, prefix=(16, 16)), 7)
    par, qo = np.asarray(inp.parent), np.asarray(inp.qo_indptr)
    for d in range(inp.path_cap):
        tl = bench.plant_accept_depth(inp, d)
        ref = oracle.greedy_accept(inp.parent, inp.draft_tokens, tl, inp.qo_indptr, inp.path_cap)
        for b in range(inp.batch):
            reach = len(_first_child_path(par, int(qo[b]), int(qo[b + 1]), d)) - 1
            assert ref.accept_len[b] == reach
