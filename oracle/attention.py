"""Oracle: tree-verify attention over a paged prefix plus the tree's own K/V.

What it computes is the plain definition ("EAGLE-2 deep dive", architecture
section: all tree tokens go through one target forward; a 2-D tree mask that
lets a node see only its causal ancestors is injected into attention;
production section: the tree mask is indexed over paged KV memory):

  for sequence b, tree node i, query head h (KV head g = h // (Hq / Hkv)):
    keys   = [prefix slots 0 .. P_b-1, read through the page table] ++ [tree nodes 0 .. N_b-1]
    allow  = prefix slot: always;  tree node j: mask[i][j]
    o[i,h] = softmax(sm_scale * q[i,h] . K^T restricted to allowed keys) @ V
    lse    = natural log of the sum of exp(scores) over allowed keys

Reading (pages silent): the verified prefix is never masked — every tree node
sees all of it; only the tree keys are filtered by the ancestor mask. This is
what the definition above implies and what "Accelerating Sonar through
speculation", EAGLE section, motivates (a custom mask over the whole sequence
is what slows attention).

All arithmetic is float64 on the given (bf16-representable or fp32) inputs. With an FP8
cache (`kv_scale` given), the pools hold E4M3 codes and a prefix key or value is the code's
value times its KV head's scale (oracle.fp8); the tree K/V stay as given.
"""

import numpy as np

from .fp8 import kv_dequantize


def _prefix_values(pool, page_table_row, length, page_size, scale):
    """Gathered prefix slots [length, heads, D] in float64, dequantised when scale is given
    (scale [heads])."""
    x = gather_prefix(pool, page_table_row, length, page_size)
    if scale is None:
        return x.astype(np.float64)
    return kv_dequantize(x, np.asarray(scale, np.float32)[None, :, None])


def gather_prefix(pool: np.ndarray, page_table_row: np.ndarray, length: int, page_size: int) -> np.ndarray:
    """Logical slots 0..length-1 of one sequence: pool[page_table[s // ps], :, s % ps, :] -> [length, Hkv, D]."""
    slots = np.arange(length)
    pages = np.asarray(page_table_row)[slots // page_size]
    if length and (pages.min() < 0 or pages.max() >= pool.shape[0]):
        raise ValueError("page table entry outside the pool")
    return pool[pages, :, slots % page_size, :]


def _one_head(qrows, K, V, allow, sm_scale):
    S = sm_scale * (qrows @ K.T)
    S = np.where(allow, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    Z = E.sum(axis=1, keepdims=True)
    O = (E / Z) @ V
    lse = (m + np.log(Z))[:, 0]
    return O, lse


def tree_verify_attention(q, k_pool, v_pool, page_table, prefix_len, k_tree, v_tree,
                          mask, qo_indptr, hq, hkv, sm_scale=None, page_size=16,
                          seqs=None, kv_scale=None):
    """Full oracle attention.

    q [T, Hq, D]; k_pool/v_pool [pages, Hkv, page_size, D]; page_table [B, max_pages];
    prefix_len [B]; k_tree/v_tree [T, Hkv, D]; mask bool [T, >= N_b] (sequence-local
    columns); qo_indptr [B+1]. Returns (o float64 [T, Hq, D], lse float64 [T, Hq]).
    `seqs` restricts the work to some sequences (other rows stay NaN). `kv_scale` [2, Hkv]
    (K scales, then V scales): the pools hold E4M3 codes.
    """
    q = np.asarray(q, np.float64)
    T, Hq, D = q.shape
    assert Hq == hq and hq % hkv == 0
    G = hq // hkv
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    qo = np.asarray(qo_indptr, np.int64)
    o = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    B = qo.shape[0] - 1
    for b in (range(B) if seqs is None else seqs):
        a, e = int(qo[b]), int(qo[b + 1])
        n = e - a
        if n == 0:
            continue
        P = int(prefix_len[b])
        Kp = _prefix_values(k_pool, page_table[b], P, page_size, None if kv_scale is None else kv_scale[0])
        Vp = _prefix_values(v_pool, page_table[b], P, page_size, None if kv_scale is None else kv_scale[1])
        K = np.concatenate([Kp, np.asarray(k_tree[a:e], np.float64)], axis=0)
        V = np.concatenate([Vp, np.asarray(v_tree[a:e], np.float64)], axis=0)
        allow = np.concatenate([np.ones((n, P), bool), np.asarray(mask[a:e, :n], bool)], axis=1)
        for h in range(Hq):
            g = h // G
            O, L = _one_head(q[a:e, h, :], K[:, g, :], V[:, g, :], allow, sm_scale)
            o[a:e, h, :] = O
            lse[a:e, h] = L
    return o, lse


def tree_verify_attention_rows(rows, q, k_pool, v_pool, page_table, prefix_len, k_tree, v_tree,
                               mask, qo_indptr, hq, hkv, sm_scale=None, page_size=16, kv_scale=None):
    """Oracle output for selected (node t, head h) rows only, one at a time.

    Used on full-size workloads where the whole oracle would take too long.
    Returns (o float64 [len(rows), D], lse float64 [len(rows)]). `kv_scale` as in
    tree_verify_attention.
    """
    q = np.asarray(q)
    D = q.shape[2]
    G = hq // hkv
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    qo = np.asarray(qo_indptr, np.int64)
    seq_of = np.searchsorted(qo, np.arange(qo[-1]), side="right") - 1
    out = np.zeros((len(rows), D))
    lses = np.zeros(len(rows))
    cache = {}
    for r, (t, h) in enumerate(rows):
        b = int(seq_of[t])
        a, e = int(qo[b]), int(qo[b + 1])
        g = h // G
        key = (b, g)
        if key not in cache:
            P = int(prefix_len[b])
            ks = None if kv_scale is None else [kv_scale[0][g]]
            vs = None if kv_scale is None else [kv_scale[1][g]]
            Kp = _prefix_values(k_pool[:, g : g + 1], page_table[b], P, page_size, ks)[:, 0]
            Vp = _prefix_values(v_pool[:, g : g + 1], page_table[b], P, page_size, vs)[:, 0]
            K = np.concatenate([Kp, np.asarray(k_tree[a:e, g], np.float64)], axis=0)
            V = np.concatenate([Vp, np.asarray(v_tree[a:e, g], np.float64)], axis=0)
            cache = {key: (K, V, P)}
        K, V, P = cache[key]
        i = t - a
        allow = np.concatenate([np.ones(P, bool), np.asarray(mask[t, : e - a], bool)])[None, :]
        O, L = _one_head(np.asarray(q[t, h], np.float64)[None, :], K, V, allow, sm_scale)
        out[r] = O[0]
        lses[r] = L[0]
    return out, lses
