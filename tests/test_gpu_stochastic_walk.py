"""GPU checks of the stochastic acceptance walk beyond the workload shapes (spec_accept through
the C ABI).

- Wide nodes: a root with more children than one listing batch holds (33-100 children, tested
  in increasing id, many rejected), on vocabularies whose slices stage with float4 loads (64,
  4096) and not (1001), exact against the oracle except sequences the oracle flags as near
  ties.
- Losslessness on the device: a root with k children whose tokens are drawn i.i.d. from the
  draft distribution q; over 2 x 10^5 sequences (four calls), the first emitted token (the
  accepted child's token or the residual bonus) must follow the target distribution p
  (chi-square p > 1e-3), as "EAGLE-2 deep dive", benchmark section, states for rejection
  sampling. The same statistic rejects a sampler that draws the bonus from p instead of the
  residual (host-side power check).
"""

import numpy as np
import pytest
import torch

import mc_accept
import oracle
from speculative_decoding_tree_parent_gb300 import binding as B

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)


def _run(parent, toks, tl, dl, u, qo, path_cap, temperature=1.0, host_logits=False):
    dev = "cuda"
    T, V = tl.shape
    Bn = len(qo) - 1
    i32 = dict(dtype=torch.int32, device=dev)
    max_nodes = int(np.diff(qo).max())
    ws = torch.zeros(B.spec_workspace_size(B.SPEC_OP_ACCEPT, Bn, T, max_nodes, 0, 0, 0, 0, V), dtype=torch.uint8,
                     device=dev)
    acc = torch.empty(Bn, **i32)
    path = torch.empty((Bn, path_cap), **i32)
    out = torch.empty((Bn, path_cap), **i32)
    flags = torch.empty(Bn, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, **i32)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    logits = (lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).pin_memory()) if host_logits else f32
    B.spec_accept(B.SPEC_STOCHASTIC, torch.from_numpy(np.asarray(parent, np.int32)).to(dev),
                  torch.from_numpy(np.asarray(toks, np.int32)).to(dev), logits(tl), torch.from_numpy(
                      np.asarray(qo, np.int32)).to(dev), max_nodes, acc, path, out, ws, draft_logits=logits(dl),
                  uniforms=f32(u), temperature=temperature, flags=flags, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return acc.cpu().numpy(), path.cpu().numpy(), out.cpu().numpy(), flags.cpu().numpy()


@pytest.mark.parametrize("V,seed", [(64, 1), (1001, 2), (4096, 3)])
def test_stochastic_wide_nodes(V, seed):
    rng = np.random.default_rng(seed)
    parents, qo = [], [0]
    for b in range(24):
        m = int(rng.integers(33, 101))          # root children: more than one batch of 32
        extra = int(rng.integers(0, 6))        # a few grandchildren under random children
        p = [-1] + [0] * m + [int(rng.integers(1, m + 1)) for _ in range(extra)]
        parents.append(p)
        qo.append(qo[-1] + len(p))
    T = qo[-1]
    tl = (rng.standard_normal((T, V)) * 2.0).astype(np.float32)
    dl = (tl + rng.standard_normal((T, V)) * 1.5).astype(np.float32)
    toks = rng.integers(0, V, T).astype(np.int32)        # mostly poor drafts: many rejections
    u = rng.random((T, 2)).astype(np.float32)
    parent = np.concatenate(parents).astype(np.int32)
    path_cap = 8
    got = _run(parent, toks, tl, dl, u, qo, path_cap)
    if V == 4096:  # the same from pinned host logits, read in place: bit for bit
        got_h = _run(parent, toks, tl, dl, u, qo, path_cap, host_logits=True)
        for x, y in zip(got, got_h):
            assert np.array_equal(x, y)
    ref = oracle.stochastic_accept(parent, toks, tl, dl, u, 1.0, np.asarray(qo), path_cap)
    keep = ref.flags == 0
    assert keep.sum() >= len(keep) - 2
    assert np.array_equal(got[0][keep], ref.accept_len[keep])
    assert np.array_equal(got[1][keep], ref.path[keep])
    assert np.array_equal(got[2][keep], ref.out_tokens[keep])


def _chisq_ok(counts, p):
    from scipy.stats import chisquare
    n = counts.sum()
    return chisquare(counts, n * p).pvalue > 1e-3


@pytest.mark.parametrize("k", [1, 3])
def test_stochastic_first_token_follows_target_on_device(k):
    per, calls = 50_000, 4          # (a launch's grid holds at most 65535 sequences)
    trials = per * calls
    p, q = mc_accept.first_token_dists(k)
    V = p.shape[0]
    rng = np.random.default_rng(7000 + k)
    n = k + 1
    parent = np.tile(np.array([-1] + [0] * k, np.int32), per)
    tl = np.tile(np.log(p).astype(np.float32), (per * n, 1))
    dl = np.tile(np.log(q).astype(np.float32), (per * n, 1))
    qo = (np.arange(per + 1) * n).astype(np.int32)
    counts = np.zeros(V, np.int64)
    accepted = 0
    for _ in range(calls):
        toks = np.zeros((per, n), np.int32)
        toks[:, 1:] = rng.choice(V, size=(per, k), p=q)
        u = rng.random((per * n, 2)).astype(np.float32)
        acc, _, out, _ = _run(parent, toks.ravel(), tl, dl, u, qo, path_cap=n)
        counts += np.bincount(out[:, 0], minlength=V)
        accepted += int((acc >= 1).sum())
    assert counts.sum() == trials
    assert _chisq_ok(counts, p)
    if k == 1:  # single draft: acceptance probability sum_x min(p(x), q(x))
        rate = accepted / trials
        want = np.minimum(p, q).sum()
        assert abs(rate - want) < 4.5 * np.sqrt(want * (1 - want) / trials)
    # power: the same statistic at this size rejects a bonus drawn from p instead of the residual
    x = rng.choice(V, size=trials, p=q)
    uu = rng.random(trials)
    wrong = np.where(uu < p[x] / q[x], x, rng.choice(V, size=trials, p=p))
    if k == 1:
        assert not _chisq_ok(np.bincount(wrong, minlength=V), p)
