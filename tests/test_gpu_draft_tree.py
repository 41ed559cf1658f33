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
