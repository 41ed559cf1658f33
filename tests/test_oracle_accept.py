"""Pins of the oracle's acceptance step.

Greedy: hand-worked golden cases; brute force over every root-to-node path on
tiny trees (a path is accepted iff each edge's token is its parent's target
argmax); the linear-draft special case; emitted count <= depth + 1.

Stochastic: hand-worked golden cases; Monte-Carlo (10^6 trials each) on a vocabulary of 8 showing
the method is lossless when draft tokens are drawn i.i.d. from the draft
distribution — the first emitted token follows p_root, the first two follow
p_root(x1) * p_x1(x2) — and the single-draft acceptance rate equals the closed
form sum_x min(p(x), q(x)).
"""

import itertools
import json
import os

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle

import mc_accept

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- greedy

def test_greedy_golden():
    g = json.load(open(os.path.join(GOLDEN, "greedy_small.json")))
    for case in g["cases"]:
        n = len(case["parent"])
        res = oracle.greedy_accept(np.array(case["parent"]), np.array(case["draft_tokens"]),
                                   np.array(case["target_logits"], np.float32), [0, n], path_cap=n)
        L = case["accept_len"]
        assert res.accept_len[0] == L, case["note"]
        assert res.path[0, : L + 1].tolist() == case["path"]
        assert res.out_tokens[0, : L + 1].tolist() == case["out_tokens"]
        assert (res.path[0, L + 1:] == -1).all() and (res.out_tokens[0, L + 1:] == -1).all()


def _tree_with_distinct_sibling_tokens(rng, n, V):
    parent = [-1]
    for i in range(1, n):
        parent.append(int(rng.integers(0, i)))
    parent = np.array(parent)
    tok = np.zeros(n, np.int64)
    tok[0] = rng.integers(0, V)
    for v in range(n):
        kids = np.flatnonzero(parent == v)
        if kids.size:
            tok[kids] = rng.choice(V, size=kids.size, replace=False)
    return parent, tok


@pytest.mark.parametrize("seed", range(40))
def test_greedy_matches_bruteforce_paths(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 12))
    V = 16
    parent, tok = _tree_with_distinct_sibling_tokens(rng, n, V)
    logits = rng.standard_normal((n, V)).astype(np.float32)
    # make matches likely: for most nodes, raise the logit of one child's token
    for v in range(n):
        kids = np.flatnonzero(parent == v)
        if kids.size and rng.random() < 0.8:
            logits[v, tok[rng.choice(kids)]] += 10
    arg = [int(np.flatnonzero(logits[v] == logits[v].max())[0]) for v in range(n)]
    # enumerate every root-to-node path; keep those whose every edge matches
    best = [0]
    for node in range(n):
        path = [node]
        while path[-1] != 0:
            path.append(int(parent[path[-1]]))
        path = path[::-1]
        ok = all(tok[path[k + 1]] == arg[path[k]] for k in range(len(path) - 1))
        if ok and len(path) > len(best):
            best = path
    res = oracle.greedy_accept(parent, tok, logits, [0, n], path_cap=n)
    L = len(best) - 1
    assert res.accept_len[0] == L
    assert res.path[0, : L + 1].tolist() == best
    want_tokens = [int(tok[c]) for c in best[1:]] + [arg[best[-1]]]
    assert res.out_tokens[0, : L + 1].tolist() == want_tokens
    depth_max = max(len(list(itertools.takewhile(lambda v: v >= 0, _ancestors(parent, i)))) for i in range(n)) - 1
    assert L + 1 <= depth_max + 1


def _ancestors(parent, i):
    v = i
    while v >= 0:
        yield v
        v = int(parent[v])


@pytest.mark.parametrize("seed", range(10))
def test_greedy_chain_is_linear_draft_case(seed):
    """A chain tree is the linear draft of "Accelerating Sonar": the accepted prefix is
    the longest run of drafts that equal the target argmax at the previous position."""
    rng = np.random.default_rng(100 + seed)
    B, V = 6, 7
    qo = [0]
    parents, toks, logits = [], [], []
    for b in range(B):
        n = int(rng.integers(1, 9))
        qo.append(qo[-1] + n)
        lg = rng.standard_normal((n, V)).astype(np.float32)
        t = rng.integers(0, V, n)
        for i in range(1, n):
            if rng.random() < 0.7:
                t[i] = int(np.argmax(lg[i - 1]))
        parents.append(np.arange(-1, n - 1))
        toks.append(t)
        logits.append(lg)
    res = oracle.greedy_accept(np.concatenate(parents), np.concatenate(toks), np.concatenate(logits), qo, 9)
    for b in range(B):
        lg, t = logits[b], toks[b]
        n = len(t)
        match = np.array([t[i] == np.argmax(lg[i - 1]) for i in range(1, n)], bool)
        L = int(np.cumprod(match).sum()) if n > 1 else 0
        assert res.accept_len[b] == L
        assert res.path[b, : L + 1].tolist() == list(range(L + 1))
        assert res.out_tokens[b, L] == int(np.argmax(lg[L]))


# ------------------------------------------------------------------------- stochastic

def test_stochastic_golden():
    g = json.load(open(os.path.join(GOLDEN, "stochastic_small.json")))
    for case in g["cases"]:
        n = len(case["parent"])
        res = oracle.stochastic_accept(
            np.array(case["parent"]), np.array(case["draft_tokens"]),
            np.log(np.array(case["target_probs"])), np.log(np.array(case["draft_probs"])),
            np.array(case["uniforms"], np.float32), g["temperature"], [0, n], path_cap=n)
        L = case["accept_len"]
        assert res.accept_len[0] == L, case["note"]
        assert res.path[0, : L + 1].tolist() == case["path"], case["note"]
        assert res.out_tokens[0, : L + 1].tolist() == case["out_tokens"], case["note"]
        assert res.flags[0] == 0


def _chisq_ok(counts, probs, alpha=1e-3):
    exp = probs * counts.sum()
    keep = exp > 0
    assert counts[~keep].sum() == 0
    return stats.chisquare(counts[keep], exp[keep]).pvalue > alpha


# Monte-Carlo pins: 10^6 trials each, in chunks run by a pool of spawned worker processes
# (the oracle is a plain per-sequence loop; the chunks only split the trials)
MC_TRIALS = 1_000_000
MC_CHUNKS = 16


def _mc_run(fn, args):
    import concurrent.futures as cf
    import multiprocessing as mp

    workers = max(1, min(len(args), os.cpu_count() or 1))
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        return list(ex.map(fn, args))


@pytest.mark.parametrize("k", [1, 2, 3])
def test_stochastic_first_token_follows_target(k):
    """Root with k children whose tokens are drawn i.i.d. from q_root: over 10^6 trials the
    first emitted token (accepted child's token, or the residual bonus) is distributed as
    p_root (chi-square p > 1e-3)."""
    per = MC_TRIALS // MC_CHUNKS
    out = _mc_run(mc_accept.first_token_chunk, [(k, per, 1000 * k + c) for c in range(MC_CHUNKS)])
    counts = sum(o[0] for o in out)
    accepted = sum(o[1] for o in out)
    p, q = mc_accept.first_token_dists(k)
    assert counts.sum() == MC_TRIALS
    assert _chisq_ok(counts, p)
    if k == 1:
        # single draft: acceptance probability sum_x min(p(x), q(x))
        rate = accepted / MC_TRIALS
        want = np.minimum(p, q).sum()
        assert abs(rate - want) < 4.5 * np.sqrt(want * (1 - want) / MC_TRIALS)


def test_stochastic_first_token_fails_without_residual():
    """Power check of the Monte-Carlo pin: a sampler that draws the bonus from p instead
    of the residual is detected by the same statistic at the same number of trials."""
    rng = np.random.default_rng(11)
    p, q = mc_accept.first_token_dists(1)
    V = p.shape[0]
    x = rng.choice(V, size=MC_TRIALS, p=q)
    u = rng.random(MC_TRIALS)
    acc = u < p[x] / q[x]
    wrong = np.where(acc, x, rng.choice(V, size=MC_TRIALS, p=p))
    assert not _chisq_ok(np.bincount(wrong, minlength=V), p)


def test_stochastic_two_tokens_joint():
    """Depth-2 trees: over 10^6 trials the first two emitted tokens follow
    p_root(x1) * p_x1(x2) (chi-square p > 1e-3); see mc_accept.joint_chunk."""
    per = MC_TRIALS // MC_CHUNKS
    joint = sum(_mc_run(mc_accept.joint_chunk, [(per, 5000 + c) for c in range(MC_CHUNKS)]))
    p_root, _, p_x, _ = mc_accept.joint_dists()
    assert joint.sum() == MC_TRIALS
    assert _chisq_ok(joint, (p_root[:, None] * p_x).ravel())


def test_stochastic_equal_distributions_accept_first_child():
    rng = np.random.default_rng(4)
    V, n = 16, 6
    parent = np.array([-1, 0, 0, 1, 1, 3])
    tl = rng.standard_normal((n, V))
    toks = rng.integers(0, V, n)
    u = rng.random((n, 2)).astype(np.float32) * 0.999
    res = oracle.stochastic_accept(parent, toks, tl, tl.copy(), u, 1.0, [0, n], path_cap=n)
    assert res.path[0, :4].tolist() == [0, 1, 3, 5]
    assert res.accept_len[0] == 3


def test_stochastic_temperature_scales_logits():
    """A root with no children emits one bonus token drawn from softmax(logits / T)."""
    rng = np.random.default_rng(8)
    V, trials, T = 8, 40000, 0.5
    lg = rng.standard_normal(V)
    res = oracle.stochastic_accept(np.full(trials, -1), np.zeros(trials, np.int64), np.tile(lg, (trials, 1)),
                                   np.tile(lg, (trials, 1)), rng.random((trials, 2)).astype(np.float32), T,
                                   np.arange(trials + 1), path_cap=1)
    assert (res.accept_len == 0).all()
    assert _chisq_ok(np.bincount(res.out_tokens[:, 0], minlength=V), softmax(lg / T))
    assert not _chisq_ok(np.bincount(res.out_tokens[:, 0], minlength=V), softmax(lg))


def test_stochastic_flags_near_ties():
    # ratio r(x)/q(x) = 0.5 exactly against u = 0.5 + 5e-7: flagged as a near tie
    p = np.array([0.5, 0.25, 0.125, 0.125])
    q = np.full(4, 0.25)
    res = oracle.stochastic_accept(np.array([-1, 0]), np.array([0, 2]), np.log(np.stack([p, p])),
                                   np.log(np.stack([q, q])), np.array([[0, 0.3], [0.5000005, 0]]),
                                   1.0, [0, 2], path_cap=2)
    assert res.flags[0] & 1
