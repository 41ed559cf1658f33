"""Attention parity inputs shared by the GPU test modules: sampled output rows, small
batches with peaked softmax, and long-prefix peaked cases. Inputs only (drawn with the
seeded generators of workloads); no verification arithmetic."""

from dataclasses import replace

import numpy as np

from speculative_decoding_tree_parent_gb300 import workloads as W


def sample_rows(inp, n, seed):
    rng = np.random.default_rng(seed)
    T, hq = inp.total_nodes, inp.hq
    rows = {(0, 0), (T - 1, hq - 1), (T - 1, 0)}
    for b in range(min(inp.batch, 8)):
        a, e = inp.qo_indptr[b], inp.qo_indptr[b + 1]
        rows.add((int(e - 1), int(rng.integers(0, hq))))
        rows.add((int(a), int(rng.integers(0, hq))))
    while len(rows) < n:
        rows.add((int(rng.integers(0, T)), int(rng.integers(0, hq))))
    return sorted(rows)


def sensitive(dtype, hq, hkv, d, prefixes, sizes, seed, scale=1.0, tree="random", q_scale=1, v_scale=1):
    """Small batch with peaked softmax (unscaled N(0,1) Q/K) and short prefixes, so the
    tree keys carry real weight and any wrong mask bit moves the output. q_scale and v_scale
    (powers of two, exact in bf16) scale Q and V: a sharper softmax for long prefixes, and
    outputs small enough that bf16's own rounding of them stays well inside 2e-2."""
    sp = W.spec(1, dtype=dtype, batch=len(prefixes), hq=hq, hkv=hkv, d=d, vocab=64, prefix=(0, 0),
                nodes=(1, 1), qkv_scale=scale, page_layout="shuffled", extra_pages=3)
    inp = W.generate(sp, seed)
    # rebuild with per-sequence prefix / tree sizes
    rng = np.random.default_rng(seed)
    parents, qo = [], [0]
    for n in sizes:
        if tree == "chain":
            p = np.arange(-1, n - 1)
        else:
            p = np.array([-1] + [int(rng.integers(max(0, i - 8), i)) for i in range(1, n)])
        parents.append(p)
        qo.append(qo[-1] + n)
    T = qo[-1]
    ps = 16
    need = [-(-(P + n) // ps) for P, n in zip(prefixes, sizes)]
    total = sum(need) + 3
    ids = rng.permutation(total)
    pt = np.full((len(sizes), max(need)), -1, np.int32)
    off = 0
    for b in range(len(sizes)):
        pt[b, : need[b]] = ids[off : off + need[b]]
        off += need[b]
    f = (lambda x: W.round_to_bf16(x)) if dtype == "bf16" else (lambda x: x)
    g = lambda *s: f((rng.standard_normal(s) * scale).astype(np.float32))
    return replace(inp, qo_indptr=np.array(qo, np.int32), parent=np.concatenate(parents).astype(np.int32),
                   draft_tokens=np.zeros(T, np.int32), q=g(T, hq, d) * np.float32(q_scale), k_tree=g(T, hkv, d),
                   v_tree=g(T, hkv, d) * np.float32(v_scale),
                   k_pool=g(total, hkv, ps, d), v_pool=g(total, hkv, ps, d) * np.float32(v_scale), page_table=pt,
                   prefix_len=np.array(prefixes, np.int32), target_logits=np.zeros((T, 64), np.float32),
                   draft_logits=None, uniforms=None, max_depth=int(max(sizes)))


# Long prefixes with peaked softmax (N(0,1) K, Q scaled by 4, V by 1/4): the key split into
# many pieces with its merge (19 splits over a 4096-token prefix, group 4), and the
# wave-model split of a batch that fills the GPU several times over (eight 32768-token
# prefixes, 128-node trees, group 8: 4 splits), checked against the per-element bound.
LONG = {
    "p4096-n64-g4": (32, 8, [4096], [64], None),
    "p32768-n128-g8-b8": (64, 8, [32768] * 8, [128] * 8, 64),
}


def long_inputs(name):
    hq, hkv, prefixes, sizes, nrows = LONG[name]
    inp = sensitive("bf16", hq, hkv, 128, prefixes, sizes, seed=300 + len(prefixes), q_scale=4,
                    v_scale=0.25)
    return inp, (None if nrows is None else sample_rows(inp, nrows, 5))
