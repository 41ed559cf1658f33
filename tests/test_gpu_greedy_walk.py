"""GPU checks of greedy acceptance walked from the root (spec_accept through the C ABI) at a
size where the library reads only the visited rows: 40 sequences of 24 nodes over a
128256-token vocabulary (streaming all 960 rows is modelled at ~86 us, the walk at ~50 us).

"EAGLE-2 deep dive", architecture section: the target's argmax at each node is contrasted with
the draft tokens and the longest accepted path is kept. The walk must give the oracle's path
and tokens bit for bit, including:
- maxima tied at several tokens in different CTAs' eighths of the row (the lowest id wins);
- rows whose maximum is zero, held by -0.0 at a low token and +0.0 at a higher one (equal
  values: the lower token wins);
- a path longer than path_cap: truncated there, SPEC_ERR_CAPACITY, the bonus taken at the
  last kept node.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_parent_gb300 import binding as B

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)

V = 128256
NB, N = 40, 24


def _inputs(seed):
    rng = np.random.default_rng(seed)
    parents, toks = [], []
    for b in range(NB):
        par, depth = [-1], [0]
        for i in range(1, N):
            cand = [u for u in range(i) if depth[u] < 8]
            p = int(rng.choice(cand))
            par.append(p)
            depth.append(depth[p] + 1)
        parents.append(par)
        toks.append(rng.integers(0, V, N))
    parent = np.concatenate(parents).astype(np.int32)
    tokens = np.concatenate(toks).astype(np.int32)
    T = NB * N
    tl = rng.standard_normal((T, V)).astype(np.float32)
    qo = (np.arange(NB + 1) * N).astype(np.int32)
    for b in range(NB):
        a = b * N
        for v in range(N):
            kids = [c for c in range(v + 1, N) if parents[b][c] == v]
            row = tl[a + v]
            kind = rng.random()
            if kids and kind < 0.6:   # the max at a child's token: the walk goes on
                row[tokens[a + int(rng.choice(kids))]] += 8.0
            elif kind < 0.75:         # a tie at three tokens in different eighths
                idx = np.sort(rng.choice(V, 3, replace=False))
                row[idx] = row.max() + 3.0
                if kids:              # a child holds the highest of the tied ids: not taken
                    tokens[a + kids[0]] = idx[2]
                    if len(kids) > 1:  # another holds the lowest: taken
                        tokens[a + kids[1]] = idx[0]
            elif kind < 0.85:         # max zero: -0.0 at a low token, +0.0 at a higher one
                row[:] = -np.abs(row) - 1.0
                lo, hi = int(rng.integers(0, V // 8)), int(rng.integers(V // 2, V))
                row[lo] = np.float32(-0.0)
                row[hi] = np.float32(0.0)
                if kids:
                    tokens[a + kids[0]] = hi
                    if len(kids) > 1 and rng.random() < 0.5:
                        tokens[a + kids[1]] = lo
    return parent, tokens, tl, qo


def _run(parent, tokens, tl, qo, path_cap):
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    T = tl.shape[0]
    ws = torch.zeros(B.spec_workspace_size(B.SPEC_OP_ACCEPT, NB, T, N, 0, 0, 0, 0, V), dtype=torch.uint8, device=dev)
    acc, path, out = torch.empty(NB, **i32), torch.empty((NB, path_cap), **i32), torch.empty((NB, path_cap), **i32)
    status = torch.zeros(1, **i32)
    B.spec_accept(B.SPEC_GREEDY, torch.from_numpy(parent).to(dev), torch.from_numpy(tokens).to(dev),
                  torch.from_numpy(tl).to(dev), torch.from_numpy(qo).to(dev), N, acc, path, out, ws, dev_status=status)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), path.cpu().numpy(), out.cpu().numpy(), int(status.item())


def test_greedy_walk_matches_oracle_with_ties_and_signed_zeros():
    parent, tokens, tl, qo = _inputs(1)
    acc, path, out, st = _run(parent, tokens, tl, qo, 9)
    assert st == 0
    ref = oracle.greedy_accept(parent, tokens, tl, qo, 9)
    assert np.array_equal(acc, ref.accept_len)
    assert np.array_equal(path, ref.path)
    assert np.array_equal(out, ref.out_tokens)
    assert (acc >= 2).sum() >= 5   # the inputs do take the walk several levels deep


def test_greedy_walk_truncates_at_path_cap():
    parent, tokens, tl, qo = _inputs(2)
    full = oracle.greedy_accept(parent, tokens, tl, qo, 9)
    cap = 3
    acc, path, out, st = _run(parent, tokens, tl, qo, cap)
    long_ = full.accept_len >= cap
    assert long_.any()
    assert st == -4 if long_.any() else st == 0   # SPEC_ERR_CAPACITY
    for b in range(NB):
        L = min(int(full.accept_len[b]), cap - 1)
        assert acc[b] == L
        assert np.array_equal(path[b, : L + 1], full.path[b, : L + 1])
        assert np.array_equal(out[b, :L], full.out_tokens[b, :L])
        last = int(full.path[b, L])
        assert out[b, L] == int(np.argmax(tl[qo[b] + last]))   # the bonus at the last kept node


def test_greedy_walk_reads_pinned_host_logits():
    """Logits in pinned host memory (read in place, only the visited rows): the same
    results as from device memory and the oracle's, for spec_accept and spec_accept_noalloc."""
    parent, tokens, tl, qo = _inputs(3)
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    T = tl.shape[0]
    ref = oracle.greedy_accept(parent, tokens, tl, qo, 9)
    host = torch.from_numpy(tl).pin_memory()
    par, tok, qo_d = (torch.from_numpy(x).to(dev) for x in (parent, tokens, qo))
    for noalloc in (False, True):
        acc, path, out = torch.empty(NB, **i32), torch.empty((NB, 9), **i32), torch.empty((NB, 9), **i32)
        status = torch.zeros(1, **i32)
        if noalloc:
            B.spec_accept_noalloc(B.SPEC_GREEDY, par, tok, host, qo_d, N, acc, path, out, dev_status=status)
        else:
            ws = torch.zeros(B.spec_workspace_size(B.SPEC_OP_ACCEPT, NB, T, N, 0, 0, 0, 0, V), dtype=torch.uint8,
                             device=dev)
            B.spec_accept(B.SPEC_GREEDY, par, tok, host, qo_d, N, acc, path, out, ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(acc.cpu().numpy(), ref.accept_len)
        assert np.array_equal(path.cpu().numpy(), ref.path)
        assert np.array_equal(out.cpu().numpy(), ref.out_tokens)


def test_accept_refuses_pageable_host_logits():
    """Logits in pageable host memory (not addressable by the device at that pointer): the
    host check answers SPEC_ERR_ARG before any launch; nothing is written."""
    import ctypes

    parent, tokens, tl, qo = _inputs(4)
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    T = tl.shape[0]
    par, tok, qo_d = (torch.from_numpy(x).to(dev) for x in (parent, tokens, qo))
    acc = torch.full((NB,), -7, **i32)
    path, out = torch.empty((NB, 9), **i32), torch.empty((NB, 9), **i32)
    ws = torch.zeros(B.spec_workspace_size(B.SPEC_OP_ACCEPT, NB, T, N, 0, 0, 0, 0, V), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, **i32)
    pageable = np.ascontiguousarray(tl)                 # plain numpy memory: never registered
    lib = B.load()
    rc = lib.spec_accept(B.SPEC_GREEDY, par.data_ptr(), tok.data_ptr(), pageable.ctypes.data, None, None,
                         ctypes.c_float(1.0), V, qo_d.data_ptr(), NB, T, N, 9, acc.data_ptr(), path.data_ptr(),
                         out.data_ptr(), None, ws.data_ptr(), ws.numel(), status.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == -1   # SPEC_ERR_ARG
    assert (acc.cpu() == -7).all() and int(status.item()) == 0
    with pytest.raises(ValueError):
        B.spec_accept(B.SPEC_GREEDY, par, tok, torch.from_numpy(pageable), qo_d, N, acc, path, out, ws)


def test_stream_reads_pinned_host_logits_unaligned_rows():
    """A 1001-token vocabulary (rows not 16-byte aligned, so the walk is unavailable): the
    streaming kernel reads every row from pinned host memory, with the oracle's results."""
    rng = np.random.default_rng(5)
    Vs, nb, n = 1001, 6, 10
    parent = np.concatenate([[-1] + [int(rng.integers(0, i)) for i in range(1, n)] for _ in range(nb)]).astype(np.int32)
    tokens = rng.integers(0, Vs, nb * n).astype(np.int32)
    tl = rng.standard_normal((nb * n, Vs)).astype(np.float32)
    qo = (np.arange(nb + 1) * n).astype(np.int32)
    for b in range(nb):                                  # a child's token at the root's argmax
        kids = [c for c in range(1, n) if parent[b * n + c] == 0]
        tl[b * n, tokens[b * n + kids[0]]] = 9.0
    ref = oracle.greedy_accept(parent, tokens, tl, qo, n)
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    acc, path, out = torch.empty(nb, **i32), torch.empty((nb, n), **i32), torch.empty((nb, n), **i32)
    status = torch.zeros(1, **i32)
    ws = torch.zeros(B.spec_workspace_size(B.SPEC_OP_ACCEPT, nb, nb * n, n, 0, 0, 0, 0, Vs), dtype=torch.uint8,
                     device=dev)
    host = torch.from_numpy(tl).pin_memory()
    B.spec_accept(B.SPEC_GREEDY, torch.from_numpy(parent).to(dev), torch.from_numpy(tokens).to(dev), host,
                  torch.from_numpy(qo).to(dev), n, acc, path, out, ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(acc.cpu().numpy(), ref.accept_len)
    assert np.array_equal(path.cpu().numpy(), ref.path)
    assert np.array_equal(out.cpu().numpy(), ref.out_tokens)
    assert (ref.accept_len >= 1).all()
