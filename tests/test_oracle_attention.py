"""Pins of the oracle's tree-verify attention.

* A chain-shaped tree's ancestor mask is the causal mask, so tree verification of
  a chain over a prefix must equal ordinary causal attention over prefix + chain
  (checked against torch's scaled_dot_product_attention, float64 on the CPU).
* A one-node tree is a plain decode step (attention over all prefix keys + itself).
* A star tree over an empty prefix: each leaf sees exactly the root and itself,
  a two-key softmax with a closed form.
* Reading the prefix through a shuffled page table changes nothing.
"""

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle


def _paged(rng, P_list, hkv, d, ps, extra=3, shuffle=True):
    """Random logical prefixes laid out in a page pool; returns pool arrays, page table
    and the logical [P, Hkv, D] views used to build the references."""
    need = [-(-max(P, 1) // ps) for P in P_list]
    total = sum(need) + extra
    ids = rng.permutation(total) if shuffle else np.arange(total)
    kp = rng.standard_normal((total, hkv, ps, d))
    vp = rng.standard_normal((total, hkv, ps, d))
    pt = np.full((len(P_list), max(need)), -1, np.int64)
    off = 0
    logical_k, logical_v = [], []
    for b, P in enumerate(P_list):
        pt[b, : need[b]] = ids[off : off + need[b]]
        off += need[b]
        slots = np.arange(P)
        logical_k.append(kp[pt[b, slots // ps], :, slots % ps, :])
        logical_v.append(vp[pt[b, slots // ps], :, slots % ps, :])
    return kp, vp, pt, logical_k, logical_v


def _sdpa(qf, kf, vf, hq, hkv, scale, causal):
    """torch reference: qf [L, Hq, D], kf/vf [S, Hkv, D] -> [L, Hq, D] (float64)."""
    G = hq // hkv
    q = torch.from_numpy(qf).permute(1, 0, 2)[None]
    k = torch.from_numpy(kf).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    v = torch.from_numpy(vf).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("P,N,hq,hkv", [(0, 5, 4, 4), (37, 1, 8, 2), (50, 9, 8, 2), (16, 4, 6, 1), (129, 7, 4, 2)])
def test_chain_equals_causal_attention(P, N, hq, hkv):
    rng = np.random.default_rng(P * 100 + N)
    d, ps = 16, 16
    kp, vp, pt, Lk, Lv = _paged(rng, [P], hkv, d, ps)
    q = rng.standard_normal((N, hq, d))
    kt = rng.standard_normal((N, hkv, d))
    vt = rng.standard_normal((N, hkv, d))
    parent = np.arange(-1, N - 1)
    mask, _ = oracle.ancestor_mask_batch(parent, [0, N])
    scale = 0.3
    o, lse = oracle.tree_verify_attention(q, kp, vp, pt, [P], kt, vt, mask, [0, N], hq, hkv,
                                          sm_scale=scale, page_size=ps)
    # causal attention over prefix + chain; the prefix positions get arbitrary queries
    qf = np.concatenate([rng.standard_normal((P, hq, d)), q], axis=0)
    kf = np.concatenate([Lk[0], kt], axis=0)
    vf = np.concatenate([Lv[0], vt], axis=0)
    ref = _sdpa(qf, kf, vf, hq, hkv, scale, causal=True)[P:]
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)
    # lse: log-sum-exp (scipy) of the allowed scores
    G = hq // hkv
    for i in range(N):
        for h in range(hq):
            s = scale * (kf[: P + i + 1, h // G, :] @ q[i, h])
            assert abs(lse[i, h] - logsumexp(s)) < 1e-10


@pytest.mark.parametrize("P", [1, 15, 16, 17, 200])
def test_single_node_is_decode(P):
    rng = np.random.default_rng(P)
    hq, hkv, d, ps = 8, 4, 32, 16
    kp, vp, pt, Lk, Lv = _paged(rng, [P], hkv, d, ps)
    q = rng.standard_normal((1, hq, d))
    kt = rng.standard_normal((1, hkv, d))
    vt = rng.standard_normal((1, hkv, d))
    mask, _ = oracle.ancestor_mask_batch([-1], [0, 1])
    o, _ = oracle.tree_verify_attention(q, kp, vp, pt, [P], kt, vt, mask, [0, 1], hq, hkv, page_size=ps)
    kf = np.concatenate([Lk[0], kt], axis=0)
    vf = np.concatenate([Lv[0], vt], axis=0)
    ref = _sdpa(q, kf, vf, hq, hkv, 1.0 / np.sqrt(d), causal=False)
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_star_tree_empty_prefix_closed_form():
    rng = np.random.default_rng(3)
    n, hq, hkv, d = 7, 2, 1, 8
    q = rng.standard_normal((n, hq, d))
    kt = rng.standard_normal((n, hkv, d))
    vt = rng.standard_normal((n, hkv, d))
    parent = [-1] + [0] * (n - 1)
    mask, _ = oracle.ancestor_mask_batch(parent, [0, n])
    kp = np.zeros((1, hkv, 16, d))
    o, lse = oracle.tree_verify_attention(q, kp, kp, np.zeros((1, 1), np.int64), [0], kt, vt, mask,
                                          [0, n], hq, hkv, sm_scale=1.0)
    for h in range(hq):
        np.testing.assert_allclose(o[0, h], vt[0, 0], rtol=1e-12)   # root sees only itself
        for i in range(1, n):
            s_root = q[i, h] @ kt[0, 0]
            s_self = q[i, h] @ kt[i, 0]
            w_root = 1.0 / (1.0 + np.exp(s_self - s_root))
            want = w_root * vt[0, 0] + (1.0 - w_root) * vt[i, 0]
            np.testing.assert_allclose(o[i, h], want, rtol=1e-10, atol=1e-12)
            assert abs(lse[i, h] - np.logaddexp(s_root, s_self)) < 1e-12


def test_page_table_layout_is_irrelevant():
    rng = np.random.default_rng(11)
    P_list, hq, hkv, d, ps = [40, 0, 77], 4, 2, 16, 8
    parents = [np.array([-1, 0, 0, 1]), np.array([-1]), np.array([-1, 0, 1, 1, 0])]
    qo = np.concatenate([[0], np.cumsum([len(p) for p in parents])])
    T = qo[-1]
    q = rng.standard_normal((T, hq, d))
    kt = rng.standard_normal((T, hkv, d))
    vt = rng.standard_normal((T, hkv, d))
    mask, _ = oracle.ancestor_mask_batch(np.concatenate(parents), qo)
    kp, vp, pt, Lk, Lv = _paged(rng, P_list, hkv, d, ps, shuffle=True)
    o1, l1 = oracle.tree_verify_attention(q, kp, vp, pt, P_list, kt, vt, mask, qo, hq, hkv, page_size=ps)
    # same logical prefixes, contiguous identity layout
    maxp = max(-(-max(P, 1) // ps) for P in P_list)
    kp2 = np.zeros((len(P_list) * maxp, hkv, ps, d))
    vp2 = np.zeros_like(kp2)
    pt2 = np.arange(len(P_list) * maxp).reshape(len(P_list), maxp)
    for b, P in enumerate(P_list):
        for s in range(P):
            kp2[pt2[b, s // ps], :, s % ps] = Lk[b][s]
            vp2[pt2[b, s // ps], :, s % ps] = Lv[b][s]
    o2, l2 = oracle.tree_verify_attention(q, kp2, vp2, pt2, P_list, kt, vt, mask, qo, hq, hkv, page_size=ps)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # row-at-a-time variant agrees with the full one
    rows = [(0, 3), (2, 1), (4, 0), (T - 1, 2), (5, 3)]
    orow, lrow = oracle.tree_verify_attention_rows(rows, q, kp, vp, pt, P_list, kt, vt, mask, qo, hq, hkv,
                                                   page_size=ps)
    for r, (t, h) in enumerate(rows):
        np.testing.assert_allclose(orow[r], o1[t, h], rtol=1e-12, atol=1e-14)
        assert abs(lrow[r] - l1[t, h]) < 1e-12


def test_tree_keys_outside_ancestry_are_invisible():
    """Changing the K/V of a node that is not an ancestor of i leaves row i unchanged;
    changing an ancestor's K/V changes it."""
    rng = np.random.default_rng(5)
    parent = np.array([-1, 0, 0, 1, 2, 3])
    n, hq, hkv, d = 6, 2, 1, 8
    mask, _ = oracle.ancestor_mask_batch(parent, [0, n])
    kp, vp, pt, _, _ = _paged(rng, [20], hkv, d, 16)
    q = rng.standard_normal((n, hq, d))
    kt = rng.standard_normal((n, hkv, d))
    vt = rng.standard_normal((n, hkv, d))
    o, _ = oracle.tree_verify_attention(q, kp, vp, pt, [20], kt, vt, mask, [0, n], hq, hkv)
    kt2, vt2 = kt.copy(), vt.copy()
    kt2[2] += 5.0
    vt2[2] -= 3.0          # node 2 is an ancestor of 4 only (and itself)
    o2, _ = oracle.tree_verify_attention(q, kp, vp, pt, [20], kt2, vt2, mask, [0, n], hq, hkv)
    for i in (0, 1, 3, 5):
        np.testing.assert_array_equal(o[i], o2[i])
    for i in (2, 4):
        assert np.abs(o[i] - o2[i]).max() > 1e-3
