"""GPU parity of the FP8 (E4M3) paged KV cache calls, through the C ABI, against the oracle.

Bars:
- attention: the per-element bound of attn_tolerance, |gpu - oracle| <= (2^-7 + 2^-12) *
  sum_k p_k |v_k| + 2^-8 |o| with the dequantised prefix values and the tree values. The
  code -> bf16 widening is exact and the scales enter P's exponent and the row sum, not
  the operands, so the bf16 path's roundings are the only error. A zeroed output and one
  missing key split must fail the same check (negative controls on the host);
- commit: the written codes bit-exact, and every other byte of the pool unchanged.
The workloads' pools are cast to codes with a per-head scale (workloads.fp8_pool); the
oracle dequantises the same codes with the same scales.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_parent_gb300 import binding as B
from speculative_decoding_tree_parent_gb300 import workloads as W
from speculative_decoding_tree_parent_gb300.step import DeviceBatch

import attn_tolerance as AT
from attn_cases import LONG, long_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)


def _check(inp, db, rows=None, controls=True):
    kc, vc, sc = db.kv_codes
    mask, _ = oracle.ancestor_mask_batch(inp.parent, inp.qo_indptr, inp.max_nodes)
    o = db.out.float().cpu().numpy().astype(np.float64)
    ref, lse, A = AT.reference(inp, mask, rows, pools=(kc, vc), kv_scale=sc)
    if rows is None:
        got, gl = o, db.lse.cpu().numpy()
    else:
        got = np.stack([o[t, h] for t, h in rows])
        gl = np.array([db.lse[t, h].item() for t, h in rows])
    err = AT.check(got, ref, A, inp.name + " (FP8 cache)")
    assert np.abs(gl - lse).max() <= 1e-3
    if controls:
        AT.negative_controls(inp, mask, ref, A, db.attn_plan()[0], rows, pools=(kc, vc), kv_scale=sc)
    return err


def _run(inp):
    db = DeviceBatch(inp, kv_fp8=True)
    db.build_mask()
    db.attention()
    torch.cuda.synchronize()
    assert db.device_status() == 0
    return db


def test_fp8_attention_llama3_single_full():
    """The Llama-3-8B-shaped single-sequence verify (4096-token prefix, 64-node tree, key
    splits + merge), every output row."""
    inp = W.generate_index(2)
    _check(inp, _run(inp))


@pytest.mark.parametrize("prefix,nodes,hq", [(0, 64, 32), (17, 5, 32), (1000, 64, 32), (4099, 130, 64),
                                             (64 * 9, 1, 8), (333, 200, 16)])
def test_fp8_attention_ragged(prefix, nodes, hq):
    """Prefixes that end inside a page and inside a 64-key block, trees over one and several
    64-key blocks, one node, no prefix, GQA groups of 1 to 8 query heads."""
    inp = W.generate(W.spec(3, batch=3, prefix=(max(0, prefix - 40), prefix), nodes=(nodes, nodes), hq=hq,
                            vocab=64, tree="random", agree_prob=0.5), seed=prefix + nodes)
    _check(inp, _run(inp))


def test_fp8_attention_batch32_sampled():
    """Batch 32, prefixes 512-8192 (the batched workload), sampled rows of every sequence."""
    inp = W.generate_index(3)
    db = _run(inp)
    rng = np.random.default_rng(0)
    rows = [(int(inp.qo_indptr[b]) + int(rng.integers(0, inp.nodes_per_seq[b])), int(rng.integers(0, inp.hq)))
            for b in range(inp.batch) for _ in range(2)]
    _check(inp, db, rows)


def test_fp8_attention_70b_32k_sampled():
    """Llama-70B-shaped 32K prefix, 8 sequences of 128 nodes (G = 8), sampled rows."""
    inp = W.generate_index(4)
    db = _run(inp)
    rng = np.random.default_rng(1)
    rows = [(int(inp.qo_indptr[b]) + int(rng.integers(0, 128)), int(rng.integers(0, inp.hq))) for b in range(8)]
    _check(inp, db, rows)


@pytest.mark.parametrize("name", sorted(LONG))
def test_fp8_attention_long_prefix_peaked(name):
    """The long-prefix peaked cases (19 key splits over 4096 tokens; the wave-model split
    of eight 32768-token prefixes) on an FP8 cache: split merge and scale folding over long
    prefixes against the per-element bound."""
    inp, rows = long_inputs(name)
    db = _run(inp)
    assert db.attn_plan()[0] >= 4
    _check(inp, db, rows)


@pytest.mark.parametrize("cfg,mode", [(2, "greedy"), (3, "greedy"), (5, "stochastic")])
def test_fp8_commit_bit_exact(cfg, mode):
    inp = W.generate_index(cfg)
    db = DeviceBatch(inp, mode=mode, kv_fp8=True)
    kc, vc, sc = db.kv_codes
    db.accept_commit(mode)
    torch.cuda.synchronize()
    assert db.device_status() == 0
    acc = db.accept_len.cpu().numpy()
    path = db.path.cpu().numpy()
    k2, v2, seq_len = oracle.kv_commit(kc, vc, inp.page_table, inp.prefix_len, inp.k_tree, inp.v_tree, path, acc,
                                       inp.qo_indptr, inp.page_size, kv_scale=sc)
    assert np.array_equal(db.k_pool.cpu().numpy(), k2)
    assert np.array_equal(db.v_pool.cpu().numpy(), v2)
    assert np.array_equal(db.seq_len.cpu().numpy(), seq_len)


def test_fp8_commit_then_attention_reads_the_new_rows():
    """A step commits its accepted rows as codes; the next attention over the longer prefix
    reads them back (the oracle sees the same committed pool)."""
    inp = W.generate_index(3)
    db = DeviceBatch(inp, kv_fp8=True)
    kc, vc, sc = db.kv_codes
    db.accept_commit("greedy")
    torch.cuda.synchronize()
    assert db.device_status() == 0
    new_len = db.seq_len.cpu().numpy()
    assert (new_len > inp.prefix_len).all()
    k2, v2 = db.k_pool.cpu().numpy(), db.v_pool.cpu().numpy()
    nxt = dataclasses.replace(inp, prefix_len=new_len.astype(np.int32))   # same pages, longer prefixes
    db2 = DeviceBatch(nxt, kv_fp8=True)
    db2.k_pool.copy_(torch.from_numpy(k2))
    db2.v_pool.copy_(torch.from_numpy(v2))
    assert np.array_equal(db2.kv_codes[2], sc)
    db2.kv_codes = (k2, v2, sc)
    db2.build_mask()
    db2.attention()
    torch.cuda.synchronize()
    assert db2.device_status() == 0
    rng = np.random.default_rng(2)
    rows = [(int(nxt.qo_indptr[b]), int(rng.integers(0, nxt.hq))) for b in range(0, nxt.batch, 4)]
    _check(nxt, db2, rows)


def test_fp8_refuses_bad_arguments():
    inp = W.generate_index(2)
    db = DeviceBatch(inp, kv_fp8=True)
    with pytest.raises(B.SpecError) as ei:
        B.spec_tree_verify_attn_kv8(db.q, db.k_pool, db.v_pool, db.kv_scale, db.page_table, db.prefix_len,
                                    db.max_prefix, db.k_tree, db.v_tree, db.mask, db.qo, db.max_nodes, db.out,
                                    ws=None)
    assert ei.value.status == -5   # the split merge needs its workspace
    lib = B.load()
    st = lib.spec_tree_verify_attn_kv8(db.q.data_ptr(), db.k_pool.data_ptr(), db.v_pool.data_ptr(), None, 1, 16,
                                       db.page_table.data_ptr(), db.page_table.shape[1], db.prefix_len.data_ptr(),
                                       db.max_prefix, db.k_tree.data_ptr(), db.v_tree.data_ptr(), db.mask.data_ptr(),
                                       db.qo.data_ptr(), 1, db.T, db.max_nodes, 32, 8, 128, 0.0, db.out.data_ptr(),
                                       None, db.attn_ws.data_ptr(), db.attn_ws.numel(), None, None)
    assert st == -1                # no kv_scale
    st = lib.spec_tree_verify_attn_kv8(db.q.data_ptr(), db.k_pool.data_ptr(), db.v_pool.data_ptr(),
                                       db.kv_scale.data_ptr(), 1, 16, db.page_table.data_ptr(),
                                       db.page_table.shape[1], db.prefix_len.data_ptr(), db.max_prefix,
                                       db.k_tree.data_ptr(), db.v_tree.data_ptr(), db.mask.data_ptr(),
                                       db.qo.data_ptr(), 1, db.T, db.max_nodes, 32, 8, 64, 0.0, db.out.data_ptr(),
                                       None, db.attn_ws.data_ptr(), db.attn_ws.numel(), None, None)
    assert st == -6                # head dim 64: no FP8 path
    with pytest.raises(B.SpecError) as ei:
        B.spec_kv_commit_kv8(db.k_tree[:, :, :8].contiguous(), db.v_tree[:, :, :8].contiguous(), db.kv_scale,
                             db.path, db.accept_len, db.qo, db.page_table, db.prefix_len, db.k_pool, db.v_pool)
    assert ei.value.status == -6   # d = 8: not a multiple of 16


def test_fp8_every_code_widens_exactly():
    """All 254 finite codes as V of a single prefix key: with q = 0 and a zero tree row the
    two keys weigh 1/2 each, so every output element is exactly value(code) / 2 (unit
    scales; bf16 holds every E4M3 value and its half). A code widened wrongly, including
    the subnormals, shows as an unequal element."""
    hkv, D = 8, 128
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    v_codes = np.resize(finite, hkv * D).reshape(hkv, D)
    k_pool = torch.zeros((1, hkv, 16, D), dtype=torch.uint8, device="cuda")
    v_pool = torch.zeros((1, hkv, 16, D), dtype=torch.uint8, device="cuda")
    v_pool[0, :, 0, :] = torch.from_numpy(v_codes).cuda()
    v_pool[0, :, 1:, :] = 0x7E   # past the prefix: never read
    z = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device="cuda")
    q, kt, vt, out = z(1, hkv, D), z(1, hkv, D), z(1, hkv, D), z(1, hkv, D)
    scale = torch.ones((2, hkv), dtype=torch.float32, device="cuda")
    mask = torch.ones((1, 1), dtype=torch.int64, device="cuda")
    i32 = lambda *v: torch.tensor(v, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(256, B.spec_workspace_size(B.SPEC_OP_ATTN, 1, 1, 1, hkv, hkv, D, 1, 0)),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.spec_tree_verify_attn_kv8(q, k_pool, v_pool, scale, i32(0).view(1, 1), i32(1), 1, kt, vt, mask, i32(0, 1), 1,
                                out, ws=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out[0].float().cpu().numpy().astype(np.float64)
    want = oracle.e4m3_decode(v_codes) / 2
    assert np.array_equal(got, want)   # (-0 and +0 compare equal: the tree's +0 is added in)
