"""Monte-Carlo trials of the stochastic-acceptance oracle, in chunks that worker processes
run (the tests sum the chunks' counts). Each chunk draws its own trees, tokens and
uniforms from its seed; the distributions under test come from fixed seeds, the same in
every chunk. Only oracle.stochastic_accept decides anything."""

import numpy as np

import oracle


def softmax(x):
    e = np.exp(x - x.max())
    return e / e.sum()


def dist(rng, V, sharp):
    return softmax(sharp * rng.standard_normal(V))


def first_token_dists(k, V=8):
    rng = np.random.default_rng(10 + k)
    return dist(rng, V, 1.0), dist(rng, V, 1.5)


def first_token_chunk(args):
    """Root with k children whose tokens are drawn i.i.d. from q_root. Returns the counts
    of the first emitted token and the number of trials that accepted a child."""
    k, trials, seed = args
    p, q = first_token_dists(k)
    V = p.shape[0]
    rng = np.random.default_rng(seed)
    n = k + 1
    parent = np.tile(np.array([-1] + [0] * k), trials)
    toks = np.zeros((trials, n), np.int64)
    toks[:, 1:] = rng.choice(V, size=(trials, k), p=q)
    tl = np.tile(np.log(p), (trials * n, 1))
    dl = np.tile(np.log(q), (trials * n, 1))
    u = rng.random((trials * n, 2)).astype(np.float32)
    qo = np.arange(trials + 1) * n
    res = oracle.stochastic_accept(parent, toks.ravel(), tl, dl, u, 1.0, qo, path_cap=n)
    return np.bincount(res.out_tokens[:, 0], minlength=V), int((res.accept_len >= 1).sum())


def joint_dists(V=6):
    rng = np.random.default_rng(21)
    p_root, q_root = dist(rng, V, 1.0), dist(rng, V, 1.0)
    p_x = np.stack([dist(rng, V, 1.0) for _ in range(V)])
    q_x = np.stack([dist(rng, V, 1.0) for _ in range(V)])
    return p_root, q_root, p_x, q_x


def joint_chunk(args):
    """Depth-2 trees (2 children per node, tokens i.i.d. from the node's draft
    distribution; a node's target and draft logits depend only on its token path). Returns
    the counts of the first two emitted tokens (x1 * V + x2); when a step emits one token,
    the second comes from the next step, a tree that is just its root."""
    trials, seed = args
    k = 2
    p_root, q_root, p_x, q_x = joint_dists()
    V = p_root.shape[0]
    rng = np.random.default_rng(seed)
    parent = [-1] + [0] * k
    for c in range(1, k + 1):
        parent += [c] * k
    parent = np.array(parent)
    n = len(parent)
    toks = np.zeros((trials, n), np.int64)
    toks[:, 1 : k + 1] = rng.choice(V, size=(trials, k), p=q_root)
    tl = np.zeros((trials, n, V))
    dl = np.zeros((trials, n, V))
    tl[:, 0], dl[:, 0] = np.log(p_root), np.log(q_root)
    for c in range(1, k + 1):
        x = toks[:, c]
        tl[:, c], dl[:, c] = np.log(p_x[x]), np.log(q_x[x])
        for j in range(k):
            gc = k + 1 + (c - 1) * k + j
            u = rng.random(trials)
            cdf = np.cumsum(q_x[x], axis=1)
            toks[:, gc] = np.minimum((cdf < u[:, None]).sum(1), V - 1)
    u = rng.random((trials * n, 2)).astype(np.float32)
    qo = np.arange(trials + 1) * n
    res = oracle.stochastic_accept(np.tile(parent, trials), toks.ravel(), tl.reshape(-1, V),
                                   dl.reshape(-1, V), u, 1.0, qo, path_cap=n)
    x1 = res.out_tokens[:, 0].copy()
    x2 = res.out_tokens[:, 1].copy()
    short = res.accept_len == 0
    m = int(short.sum())
    nxt = oracle.stochastic_accept(np.full(m, -1), np.zeros(m, np.int64), np.log(p_x[x1[short]]),
                                   np.log(p_x[x1[short]]), rng.random((m, 2)).astype(np.float32),
                                   1.0, np.arange(m + 1), path_cap=1)
    x2[short] = nxt.out_tokens[:, 0]
    return np.bincount(x1 * V + x2, minlength=V * V)
