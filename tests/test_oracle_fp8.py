"""Pins of the oracle's E4M3 codec and of the FP8 KV cache's use of it in attention and
commit.

The codec is pinned against:
- values the OCP 8-bit floating-point format fixes (largest normal 448, smallest normal
  2^-6, largest subnormal 7/8 * 2^-6, smallest subnormal 2^-9, 1.0, the NaN codes);
- an independent implementation, torch's float8_e4m3fn cast (round to nearest even, inside
  the range where that cast does not overflow to NaN);
- brute force over all 256 codes.

The FP8 attention and commit are pinned to the plain (already pinned) oracle over pools that
torch's float8 decode dequantises."""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as F


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_format_values():
    d = F.e4m3_decode(np.array([0x7E, 0x08, 0x07, 0x01, 0x38, 0x00, 0x80, 0xFE, 0x40], np.uint8))
    assert d.tolist()[:5] == [448.0, 2.0 ** -6, 0.875 * 2.0 ** -6, 2.0 ** -9, 1.0]
    assert d[5] == 0.0 and not np.signbit(d[5])
    assert d[6] == 0.0 and np.signbit(d[6])
    assert d[7] == -448.0 and d[8] == 2.0
    assert np.isnan(F.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    a, b = F.e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    ok = ~np.isnan(a)
    assert np.array_equal(a[ok], b[ok]) and np.array_equal(np.signbit(a[ok]), np.signbit(b[ok]))


def test_decode_is_increasing_and_symmetric():
    g = F.e4m3_decode(np.arange(127, dtype=np.uint8))
    assert np.all(np.diff(g) > 0)
    assert np.array_equal(F.e4m3_decode(np.arange(127, dtype=np.uint8) | 0x80), -g)


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    g = F.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = ((g[1:] + g[:-1]) / 2).astype(np.float32)        # exact ties (fp32 holds them)
    assert np.array_equal(mids.astype(np.float64), (g[1:] + g[:-1]) / 2)
    x = np.concatenate([
        g.astype(np.float32), mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
        (rng.standard_normal(20000) * 30).astype(np.float32),
        (rng.standard_normal(20000) * 2.0 ** -7).astype(np.float32),
        np.float32([463.9, -463.9, 1e-12, -1e-12, 0.0, -0.0]),
    ])
    x = np.concatenate([x, -x])
    assert np.array_equal(F.e4m3_encode(x), _torch_encode(x))


def test_encode_is_nearest_by_brute_force():
    rng = np.random.default_rng(1)
    x = np.concatenate([(rng.standard_normal(3000) * 40).astype(np.float32), np.float32([600.0, -1e5])])
    codes = F.e4m3_encode(x)
    allv = F.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = np.where(np.isnan(allv), np.inf, allv)
    for xi, c in zip(x.tolist(), codes.tolist()):
        xs = min(max(xi, -448.0), 448.0)                  # saturation of finite values
        best = np.min(np.abs(fin - xs))
        assert abs(allv[c] - xs) == best


def test_encode_ties_go_to_even_and_saturation():
    # 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39): even code 0x38;
    # 1.1875 halfway between 1.125 (0x39) and 1.25 (0x3A): 0x3A
    assert F.e4m3_encode(np.float32([1.0625, 1.1875, -1.0625])).tolist() == [0x38, 0x3A, 0xB8]
    assert F.e4m3_encode(np.float32([449.0, 464.0, 1e30, np.inf, -500.0])).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert F.e4m3_encode(np.float32([np.nan]))[0] & 0x7F == 0x7F
    # round trip of every finite code
    c = np.array([i for i in range(256) if (i & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(F.e4m3_encode(F.e4m3_decode(c).astype(np.float32)), c)


def test_kv_quantize_divides_in_fp32():
    x = np.float32([3.0, -7.5, 0.3])
    s = np.float32(0.7)
    assert np.array_equal(F.kv_quantize(x, s), _torch_encode(x / s))


def _fp8_case(seed, B=2, hq=4, hkv=2, D=16, ps=4, P=(9, 0), N=(5, 3)):
    rng = np.random.default_rng(seed)
    qo = np.concatenate([[0], np.cumsum(N)]).astype(np.int32)
    T = int(qo[-1])
    parent = np.concatenate([[-1] + [int(rng.integers(0, i)) for i in range(1, n)] for n in N]).astype(np.int32)
    mask, _ = oracle.ancestor_mask_batch(parent, qo, max(N))
    pages_per = max(1, -(-max(P) // ps))
    n_pages = B * pages_per + 1
    page_table = rng.permutation(n_pages)[: B * pages_per].reshape(B, pages_per).astype(np.int32)
    kc = rng.integers(0, 256, (n_pages, hkv, ps, D)).astype(np.uint8)
    vc = rng.integers(0, 256, (n_pages, hkv, ps, D)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x3C   # no NaN codes in a cache
    vc[(vc & 0x7F) == 0x7F] = 0x3C
    scale = np.float32(rng.uniform(0.01, 0.1, (2, hkv)))
    q = rng.standard_normal((T, hq, D))
    kt = rng.standard_normal((T, hkv, D))
    vt = rng.standard_normal((T, hkv, D))
    return q, kc, vc, scale, page_table, np.array(P, np.int32), kt, vt, mask, qo, hq, hkv, ps


def test_fp8_attention_is_attention_over_the_dequantised_pool():
    q, kc, vc, scale, pt, P, kt, vt, mask, qo, hq, hkv, ps = _fp8_case(2)
    o8, l8 = oracle.tree_verify_attention(q, kc, vc, pt, P, kt, vt, mask, qo, hq, hkv, page_size=ps,
                                          kv_scale=scale)
    kd = _torch_decode(kc) * scale[0].astype(np.float64)[None, :, None, None]
    vd = _torch_decode(vc) * scale[1].astype(np.float64)[None, :, None, None]
    o, l = oracle.tree_verify_attention(q, kd, vd, pt, P, kt, vt, mask, qo, hq, hkv, page_size=ps)
    np.testing.assert_allclose(o8, o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l8, l, rtol=1e-13)
    rows = [(0, 0), (3, 3), (6, 1), (7, 2)]
    orow, lrow = oracle.tree_verify_attention_rows(rows, q, kc, vc, pt, P, kt, vt, mask, qo, hq, hkv,
                                                   page_size=ps, kv_scale=scale)
    for r, (t, h) in enumerate(rows):
        np.testing.assert_allclose(orow[r], o[t, h], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lrow[r], l[t, h], rtol=1e-13)


def test_fp8_commit_writes_quantised_rows_only():
    rng = np.random.default_rng(3)
    hkv, D, ps = 2, 8, 4
    kc = rng.integers(0, 126, (6, hkv, ps, D)).astype(np.uint8)
    vc = rng.integers(0, 126, (6, hkv, ps, D)).astype(np.uint8)
    pt = np.array([[4, 1, 3]], np.int32)
    kt = (rng.standard_normal((5, hkv, D)) * 3).astype(np.float32)
    vt = (rng.standard_normal((5, hkv, D)) * 3).astype(np.float32)
    scale = np.float32([[0.02, 0.5], [0.03, 0.25]])
    path = np.array([[0, 2, 4]], np.int32)
    kp, vp, seq_len = oracle.kv_commit(kc, vc, pt, np.int32([3]), kt, vt, path, np.int32([2]),
                                       np.int32([0, 5]), page_size=ps, kv_scale=scale)
    assert seq_len.tolist() == [6]
    touched = np.zeros(kc.shape, bool)
    for i, node in enumerate([0, 2, 4]):
        slot = 3 + i
        page, r = pt[0, slot // ps], slot % ps
        touched[page, :, r, :] = True
        for g in range(hkv):
            assert np.array_equal(kp[page, g, r], _torch_encode(kt[node, g] / scale[0, g]))
            assert np.array_equal(vp[page, g, r], _torch_encode(vt[node, g] / scale[1, g]))
    assert np.array_equal(kp[~touched], kc[~touched]) and np.array_equal(vp[~touched], vc[~touched])


def test_workload_fp8_pool_is_the_pool_in_codes():
    """The generator's FP8 pools (test data): no NaN codes, one positive scale per KV head
    for K and for V (max|x| / 448), and every dequantised value within E4M3 rounding
    (half a unit in the last place: relative 2^-4, or 2^-10 absolute near zero) of the
    bf16 pool it came from."""
    from speculative_decoding_tree_parent_gb300 import workloads as W
    inp = W.generate(W.spec(3, batch=2, prefix=(100, 300), nodes=(8, 8), vocab=64, tree="random",
                            agree_prob=0.5), seed=4)
    kc, vc, sc = W.fp8_pool(inp)
    assert kc.shape == inp.k_pool.shape and kc.dtype == np.uint8 and vc.dtype == np.uint8
    assert sc.shape == (2, inp.hkv) and (sc > 0).all()
    for codes, pool, s in ((kc, inp.k_pool, sc[0]), (vc, inp.v_pool, sc[1])):
        assert not ((codes & 0x7F) == 0x7F).any()
        x = pool.astype(np.float64) / s.astype(np.float64)[None, :, None, None]
        d = F.e4m3_decode(codes)
        assert np.all(np.abs(d - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10) * 1.0001)
        assert np.isclose(np.abs(x).max(), 448.0, rtol=1e-6)
