"""GPU parity of the device-side EAGLE-2 draft tree (spec_tree_init / spec_tree_expand,
through the C ABI) against the oracle's priority-queue construction.

Bars: parent and token arrays and node counts exact, except sequences in which the oracle
saw a pop whose best two confidences were within a relative 1e-6 (fp32 probabilities on
the GPU may order those either way); those are counted and must stay rare. Exact ties
(identical logits at depth 1) are decided identically and compared too.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_parent_gb300 import binding as B

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)


def _build_gpu(logits_all, roots, n, k, depth, threshold=0.0):
    """Run a whole construction on the device: init, then n - 1 expansions (a call on a
    completed tree does nothing), the draft rows read from logits_all[b][node]."""
    Bn, N, V = logits_all.shape
    assert N >= n
    dev = logits_all.device
    state = torch.zeros(B.spec_workspace_size(B.SPEC_OP_TREE, Bn, 0, n, 0, 0, 0, 0, 0), dtype=torch.uint8,
                        device=dev)
    parent = torch.empty((Bn, n), dtype=torch.int32, device=dev)
    tokens = torch.empty((Bn, n), dtype=torch.int32, device=dev)
    nn = torch.empty(Bn, dtype=torch.int32, device=dev)
    nxt = torch.empty(Bn, dtype=torch.int32, device=dev)
    flags = torch.empty(Bn, dtype=torch.uint8, device=dev)
    B.spec_tree_init(roots, n, state, parent, tokens, nn, nxt, flags)
    for _ in range(n - 1):
        B.spec_tree_expand(logits_all, n, k, depth, state, parent, tokens, nn, nxt, row_stride=N * V,
                           node_stride=V, threshold=threshold, flags=flags)
    torch.cuda.synchronize()
    return parent.cpu().numpy(), tokens.cpu().numpy(), nn.cpu().numpy(), nxt.cpu().numpy(), flags.cpu().numpy()


def _compare(logits, roots, n, k, depth, threshold=0.0, strict=False):
    Bn = logits.shape[0]
    dev = torch.from_numpy(logits).cuda()
    parent, tokens, nn, nxt, flags = _build_gpu(dev, torch.from_numpy(roots).cuda(), n, k, depth, threshold)
    assert (nxt == -1).all()
    tight = 0
    for b in range(Bn):
        p, t, s, is_tight = oracle.best_first_tree(lambda u: logits[b, u], int(roots[b]), n, k, depth, threshold)
        if is_tight and not strict:
            tight += 1
            continue
        assert nn[b] == len(p), b
        assert np.array_equal(parent[b, : len(p)], p), b
        assert np.array_equal(tokens[b, : len(p)], t), b
        assert (parent[b, len(p):] == -1).all() and (tokens[b, len(p):] == -1).all()
    return tight, parent, tokens, nn


def test_tree_llama3_vocab_top10_depth8():
    """The shape the verification workloads use: 128256-token vocabulary, top-10, depth 8,
    64 nodes, draft logits ~ N(0, 2^2)."""
    rng = np.random.default_rng(11)
    V, n = 128256, 64
    logits = (rng.standard_normal((1, n, V)) * 2.0).astype(np.float32)
    tight, *_ = _compare(logits, np.array([17], np.int32), n, 10, 8)
    assert tight == 0


@pytest.mark.parametrize("seed,k,depth,n", [(1, 10, 8, 64), (2, 4, 6, 48), (3, 16, 3, 128), (4, 1, 8, 9)])
def test_tree_batch(seed, k, depth, n):
    rng = np.random.default_rng(seed)
    Bn, V = 3, 4096
    logits = (rng.standard_normal((Bn, n, V)) * 3.0).astype(np.float32)
    roots = rng.integers(0, V, Bn).astype(np.int32)
    tight, parent, tokens, nn = _compare(logits, roots, n, k, depth)
    assert tight <= 1
    # the trees feed the mask call directly (every tree full: sequence b = rows b*n .. b*n+n-1)
    if (nn == n).all():
        par = torch.from_numpy(parent.reshape(-1)).cuda()
        qo = torch.arange(0, (Bn + 1) * n, n, dtype=torch.int32, device="cuda")
        words = (n + 63) // 64
        mask = torch.zeros((Bn * n, words), dtype=torch.int64, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.spec_build_tree_mask(par, qo, n, mask, None, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        m, _ = oracle.ancestor_mask_batch(parent.reshape(-1), qo.cpu().numpy(), n)
        assert np.array_equal(mask.cpu().numpy().view(np.uint64), oracle.pack_mask_words(m, words))


def test_tree_threshold_and_small_vocab():
    """A threshold that leaves the queue empty before the budget: fewer nodes, exact."""
    rng = np.random.default_rng(5)
    Bn, V, n = 4, 100, 32
    logits = (rng.standard_normal((Bn, n, V)) * 1.5).astype(np.float32)
    roots = np.arange(Bn, dtype=np.int32)
    tight, parent, tokens, nn = _compare(logits, roots, n, 3, 5, threshold=0.05)
    assert (nn < n).any()


def test_tree_exact_ties_at_depth_one():
    """Quantised logits: equal logits tie in the top-k (lower token id first) and give equal
    confidences (the earlier push first); at depth 1 both sides compute the same products."""
    rng = np.random.default_rng(6)
    Bn, V, n = 5, 64, 9
    logits = rng.integers(0, 3, (Bn, n, V)).astype(np.float32)
    roots = np.zeros(Bn, np.int32)
    _compare(logits, roots, n, 8, 1, strict=True)


def test_tree_refuses_bad_arguments():
    dev = "cuda"
    state = torch.zeros(16, dtype=torch.uint8, device=dev)   # too small
    z = torch.zeros((1, 4), dtype=torch.int32, device=dev)
    one = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(B.SpecError) as ei:
        B.spec_tree_init(one, 4, state, z, z, one, one)
    assert ei.value.status == -5
    big = torch.zeros(B.spec_workspace_size(B.SPEC_OP_TREE, 1, 0, 4, 0, 0, 0, 0, 0), dtype=torch.uint8, device=dev)
    logits = torch.zeros((1, 4, 8), dtype=torch.float32, device=dev)
    with pytest.raises(B.SpecError) as ei:
        B.spec_tree_expand(logits, 4, 17, 2, big, z, z, one, one, row_stride=32, node_stride=8)  # topk > 16
    assert ei.value.status == -1


# ---------------------------------------------------------------- the multi-row call
from draft_protocol import EdgeRows, multi_row_tree  # noqa: E402


def _build_multi(er, roots, n, k, depth, width, threshold=0.0):
    """Drive spec_tree_expand_multi to completion, the host standing in for the draft model:
    after each call it writes the rows of the listed requests (EdgeRows, keyed by parent and
    token). Returns the device outputs and, per call, every sequence's request list."""
    Bn, V = len(roots), er.vocab
    dev = "cuda"
    state = torch.zeros(B.spec_workspace_size(B.SPEC_OP_TREE, Bn, 0, n, 0, 0, 0, 0, 0), dtype=torch.uint8,
                        device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    parent, tokens = torch.empty((Bn, n), **i32), torch.empty((Bn, n), **i32)
    nn, nxt, req_n = torch.empty(Bn, **i32), torch.empty(Bn, **i32), torch.empty(Bn, **i32)
    req_p, req_t = torch.empty((Bn, width), **i32), torch.empty((Bn, width), **i32)
    flags = torch.empty(Bn, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, **i32)
    B.spec_tree_init(torch.from_numpy(roots).cuda(), n, state, parent, tokens, nn, nxt, flags)
    rows = torch.zeros((Bn, width, V), dtype=torch.float32, device=dev)
    host = np.zeros((Bn, width, V), np.float32)
    reqs = [[(-1, int(roots[b]))] if n > 1 else [] for b in range(Bn)]
    calls = []
    while any(reqs):
        host[:] = 0
        for b in range(Bn):
            for j, (p, t) in enumerate(reqs[b]):
                host[b, j] = er.row(b, p, t)
        rows.copy_(torch.from_numpy(host))
        B.spec_tree_expand_multi(rows, n, k, depth, state, parent, tokens, nn, nxt, req_p, req_t, req_n,
                                 threshold=threshold, flags=flags, dev_status=status)
        calls.append(reqs)
        rn, rp, rt = req_n.cpu().numpy(), req_p.cpu().numpy(), req_t.cpu().numpy()
        reqs = [[(int(rp[b, j]), int(rt[b, j])) for j in range(rn[b])] for b in range(Bn)]
        for b in range(Bn):
            assert (rp[b, rn[b]:] == -1).all() and (rt[b, rn[b]:] == -1).all()
        assert len(calls) <= n + 1
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return (parent.cpu().numpy(), tokens.cpu().numpy(), nn.cpu().numpy(), nxt.cpu().numpy(), flags.cpu().numpy(),
            calls)


def _compare_multi(er, roots, n, k, depth, width, threshold=0.0, strict=False):
    parent, tokens, nn, nxt, flags, calls = _build_multi(er, roots, n, k, depth, width, threshold)
    assert (nxt == -1).all()
    tight = 0
    for b in range(len(roots)):
        p, t, s, is_tight = oracle.best_first_tree(er.of(b), int(roots[b]), n, k, depth, threshold, row_key="edge")
        if is_tight and not strict:
            tight += 1
            continue
        assert nn[b] == len(p), b
        assert np.array_equal(parent[b, : len(p)], p), b
        assert np.array_equal(tokens[b, : len(p)], t), b
        assert (parent[b, len(p):] == -1).all() and (tokens[b, len(p):] == -1).all()
        # the requests, call by call, are the protocol's (the host model in fp64)
        model = multi_row_tree(er.of(b), int(roots[b]), n, k, depth, width, threshold)
        got = [c[b] for c in calls if c[b]]
        assert got == model.requests, b
    return tight, len(calls)


@pytest.mark.parametrize("width", [1, 4, 8])
def test_multi_tree_llama3_vocab(width):
    """128256-token vocabulary, top-10, depth 8, 64 nodes, draft logits ~ N(0, 2^2): the
    one-row construction's tree, the protocol's requests, and (width 8) 9 calls instead of 63."""
    er = EdgeRows(21, 128256, scale=2.0)
    tight, ncalls = _compare_multi(er, np.array([17], np.int32), 64, 10, 8, width)
    assert tight == 0
    assert ncalls == {1: 63, 4: 17, 8: 9}[width]


@pytest.mark.parametrize("seed,V,k,depth,n,width,bump", [
    (1, 4096, 10, 8, 64, 8, 0.0), (2, 4096, 4, 6, 48, 3, 0.0), (3, 4096, 16, 3, 128, 8, 0.0),
    (4, 4096, 1, 8, 9, 8, 0.0), (5, 1001, 10, 8, 64, 8, 12.0), (6, 4096, 10, 8, 64, 8, 14.0)])
def test_multi_tree_batch(seed, V, k, depth, n, width, bump):
    """Three sequences per call; odd vocabulary (scalar loads); confident draft heads
    (bump: deep chains, where fewer candidates are popped per call)."""
    rng = np.random.default_rng(seed)
    roots = rng.integers(0, V, 3).astype(np.int32)
    er = EdgeRows(100 + seed, V, scale=2.0, bump=bump)
    tight, _ = _compare_multi(er, roots, n, k, depth, width)
    assert tight <= 1


def test_multi_tree_threshold_and_ties():
    """A threshold that empties the queue before the budget; quantised logits (exact ties in
    the top-k and equal confidences at depth 1)."""
    er = EdgeRows(7, 100, scale=1.5)
    _compare_multi(er, np.arange(4, dtype=np.int32), 32, 3, 5, 8, threshold=0.05)

    class Quantised(EdgeRows):
        def row(self, b, parent, token):
            r = super().row(b, parent, token)
            return np.floor(np.abs(r)).astype(np.float32)

    _compare_multi(Quantised(8, 64, scale=1.2), np.zeros(5, np.int32), 9, 8, 1, 8, strict=True)


def test_multi_tree_edges():
    """max_nodes 1 (nothing to request, a call changes nothing); a width above 8 is refused on
    the host; a call narrower than the pending request list is refused on the device and
    leaves the tree as it was."""
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    st1 = torch.zeros(B.spec_workspace_size(B.SPEC_OP_TREE, 1, 0, 1, 0, 0, 0, 0, 0), dtype=torch.uint8, device=dev)
    par, tok = torch.empty((1, 1), **i32), torch.empty((1, 1), **i32)
    nn, nxt, rn = torch.full((1,), 7, **i32), torch.empty(1, **i32), torch.full((1,), 5, **i32)
    rp, rt = torch.full((1, 2), 9, **i32), torch.full((1, 2), 9, **i32)
    B.spec_tree_init(torch.tensor([3], **i32), 1, st1, par, tok, nn, nxt)
    rows = torch.zeros((1, 2, 64), dtype=torch.float32, device=dev)
    B.spec_tree_expand_multi(rows, 1, 4, 4, st1, par, tok, nn, nxt, rp, rt, rn)
    torch.cuda.synchronize()
    assert int(nn.item()) == 1 and int(nxt.item()) == -1 and int(rn.item()) == 5   # skipped: untouched

    with pytest.raises(B.SpecError) as ei:
        B.spec_tree_expand_multi(torch.zeros((1, 9, 64), dtype=torch.float32, device=dev), 1, 4, 4, st1, par, tok,
                                 nn, nxt, torch.empty((1, 9), **i32), torch.empty((1, 9), **i32), rn)
    assert ei.value.status == -1

    er = EdgeRows(9, 256, scale=2.0)
    n = 16
    st = torch.zeros(B.spec_workspace_size(B.SPEC_OP_TREE, 1, 0, n, 0, 0, 0, 0, 0), dtype=torch.uint8, device=dev)
    par, tok = torch.empty((1, n), **i32), torch.empty((1, n), **i32)
    rp8, rt8 = torch.empty((1, 8), **i32), torch.empty((1, 8), **i32)
    status = torch.zeros(1, **i32)
    B.spec_tree_init(torch.tensor([1], **i32), n, st, par, tok, nn, nxt)
    rows8 = torch.zeros((1, 8, 256), dtype=torch.float32, device=dev)
    rows8[0, 0] = torch.from_numpy(er.row(0, -1, 1))
    B.spec_tree_expand_multi(rows8, n, 4, 4, st, par, tok, nn, nxt, rp8, rt8, rn, dev_status=status)
    torch.cuda.synchronize()
    listed = int(rn.item())
    assert listed > 2 and int(status.item()) == 0
    before = (par.clone(), tok.clone(), int(nn.item()))
    rp2, rt2 = torch.empty((1, 2), **i32), torch.empty((1, 2), **i32)
    B.spec_tree_expand_multi(torch.zeros((1, 2, 256), dtype=torch.float32, device=dev), n, 4, 4, st, par, tok, nn,
                             nxt, rp2, rt2, rn, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -1
    assert torch.equal(par, before[0]) and torch.equal(tok, before[1]) and int(nn.item()) == before[2]
    assert int(rn.item()) == listed


def test_multi_tree_many_sequences():
    """Twenty sequences at width 8: 1280 CTAs, more than one wave, so a sequence's replaying
    cluster may start after other sequences' clusters have finished (nothing waits)."""
    rng = np.random.default_rng(31)
    roots = rng.integers(0, 4096, 20).astype(np.int32)
    er = EdgeRows(131, 4096, scale=2.5)
    tight, ncalls = _compare_multi(er, roots, 32, 4, 6, 8)
    assert tight <= 2
