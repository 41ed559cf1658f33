"""CPU checks that the seeded synthetic workloads have the structure their recipes state
(the inputs the bench and the parity tests run on): batch, heads, prefix ranges, page
layout, node budgets, depth and branching limits, tree shape, and the draws' distributions.
Dimensions no checked property depends on (head dim, head counts, vocabulary) are shrunk
where the full size would take more than a few seconds on the host."""

import numpy as np

from speculative_decoding_tree_parent_gb300 import workloads as W


def _trees(inp):
    qo, par = np.asarray(inp.qo_indptr), np.asarray(inp.parent)
    for b in range(inp.batch):
        a, e = int(qo[b]), int(qo[b + 1])
        p = par[a:e]
        assert p[0] == -1
        assert all(0 <= p[i] < i for i in range(1, e - a))   # parents precede children
        depth = np.zeros(e - a, int)
        for i in range(1, e - a):
            depth[i] = depth[p[i]] + 1
        yield b, a, p, depth


def _pages(inp):
    pt, P, qo = np.asarray(inp.page_table), np.asarray(inp.prefix_len), np.asarray(inp.qo_indptr)
    used = []
    for b in range(inp.batch):
        need = -(-(int(P[b]) + int(qo[b + 1] - qo[b])) // inp.page_size)   # prefix + tree slots
        row = pt[b, :need]
        assert (row >= 0).all() and (row < inp.num_pages).all()
        used.append(row)
    flat = np.concatenate(used)
    assert len(np.unique(flat)) == len(flat)   # no page shared between sequences or slots
    return used


def _bf16(x):
    return ((np.ascontiguousarray(x, np.float32).view(np.uint32) & 0xFFFF) == 0).all()


def test_workload1_tiny_fp32():
    inp = W.generate_index(1)
    assert (inp.batch, inp.hq, inp.hkv, inp.d, inp.vocab) == (1, 4, 1, 64, 1000)
    assert inp.prefix_len.tolist() == [128] and inp.max_nodes == 16
    (row,) = _pages(inp)
    assert row.tolist() == list(range(len(row)))   # identity page table
    for _, _, p, depth in _trees(inp):
        assert depth.max() <= 4
    many = W.generate(W.spec(1, batch=100), 1)      # the 0.7 agreement rate, over 1500 nodes
    tl, tok, par, qo = many.target_logits, many.draft_tokens, many.parent, many.qo_indptr
    agree = [tok[a + i] == np.argmax(tl[a + par[a + i]]) for b in range(many.batch)
             for a in [int(qo[b])] for i in range(1, int(qo[b + 1]) - a)]
    assert 0.65 < np.mean(agree) < 0.75


def test_workload2_single_sequence_llama3_8b():
    inp = W.generate_index(2)
    assert (inp.batch, inp.hq, inp.hkv, inp.d, inp.vocab, inp.page_size) == (1, 32, 8, 128, 128256, 16)
    assert inp.prefix_len.tolist() == [4096] and inp.max_nodes == 64
    (row,) = _pages(inp)
    assert sorted(row.tolist()) != row.tolist()    # shuffled page table
    for _, a, p, depth in _trees(inp):
        assert depth.max() <= 8
        assert np.bincount(p[1:]).max() <= 10       # top-10 expansion
        for v in range(len(p)):                     # siblings carry distinct tokens
            kids = np.flatnonzero(p == v)
            assert len(set(inp.draft_tokens[a + kids].tolist())) == len(kids)
    assert _bf16(inp.q) and _bf16(inp.k_tree) and _bf16(inp.k_pool)
    assert abs(inp.q.std() * np.sqrt(128.0) - 1.0) < 0.05          # N(0, 1) / sqrt(128)
    assert abs(inp.target_logits.mean()) < 0.01 and abs(inp.target_logits.std() - 1.0) < 0.01


def test_workload2_bump_rate():
    """+4 on the first child's token with probability 0.8: that logit exceeds 2 for about
    0.8 x P(N(4,1) > 2) + 0.2 x P(N(0,1) > 2) = 0.79 of the non-leaf nodes."""
    inp = W.generate(W.spec(2, batch=24, vocab=4096, hq=8, hkv=8, d=16, prefix=(16, 16)), 2)
    hits = []
    for _, a, p, _ in _trees(inp):
        for v in range(len(p)):
            kids = np.flatnonzero(p == v)
            if kids.size:
                hits.append(inp.target_logits[a + v, inp.draft_tokens[a + kids.min()]] > 2.0)
    assert len(hits) > 150 and 0.70 < np.mean(hits) < 0.87


def test_workload3_batch32_scattered_pages():
    inp = W.generate(W.spec(3, hq=4, hkv=1, d=16, vocab=256), 3)
    assert inp.batch == 32 and inp.max_nodes == 64 and (np.diff(inp.qo_indptr) == 64).all()
    P = np.asarray(inp.prefix_len)
    assert P.min() >= 512 and P.max() <= 8192 and P.max() - P.min() > 2000
    rows = _pages(inp)
    assert sum(sorted(r.tolist()) != r.tolist() for r in rows) >= 30   # pages scattered
    for _, _, p, depth in _trees(inp):
        assert depth.max() <= 8 and np.bincount(p[1:]).max() <= 10


def test_workload4_70b_stochastic():
    inp = W.generate(W.spec(4, hq=8, hkv=1, d=16, vocab=2048), 4)
    assert inp.batch == 8 and (np.asarray(inp.prefix_len) == 32768).all() and inp.max_nodes == 128
    assert inp.modes == ("stochastic",) and inp.temperature == 1.0
    noise = inp.draft_logits - inp.target_logits
    assert abs(noise.std() - 0.5) < 0.01 and abs(noise.mean()) < 0.01   # draft = target + N(0, 0.5^2)
    assert inp.uniforms.shape == (inp.total_nodes, 2)
    assert (inp.uniforms >= 0).all() and (inp.uniforms < 1).all()
    for _, a, p, depth in _trees(inp):
        assert depth.max() <= 8 and np.bincount(p[1:]).max() <= 10
        for c in range(1, len(p)):   # children come from the parent's own draft top-10
            top = np.argsort(-inp.draft_logits[a + p[c]], kind="stable")[:10]
            assert inp.draft_tokens[a + c] in top


def test_workload5_chains():
    inp = W.generate(W.spec(5, hq=8, hkv=1, d=16, vocab=1024), 5)
    assert inp.batch == 128 and set(inp.modes) == {"greedy", "stochastic"}
    n = np.diff(inp.qo_indptr)
    assert n.min() >= 2 and n.max() <= 9 and len(set(n.tolist())) >= 6   # 1-8 draft tokens
    P = np.asarray(inp.prefix_len)
    assert P.min() >= 256 and P.max() <= 4096
    for _, a, p, _ in _trees(inp):
        assert p.tolist() == list(range(-1, len(p) - 1))   # a chain
        for i in range(1, len(p)):                          # the draft's top-1 token
            assert inp.draft_tokens[a + i] == np.argmax(inp.draft_logits[a + i - 1])
    _pages(inp)
