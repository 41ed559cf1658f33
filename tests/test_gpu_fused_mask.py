"""GPU parity of spec_tree_verify_attn_parents: the attention call that builds its ancestor
bits from the parent array must give bit for bit what spec_build_tree_mask followed by
spec_tree_verify_attn gives (the same arithmetic, only the bits' source differs). It is also
checked against the oracle directly, and a parent array that is not a tree must be
reported."""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_parent_gb300 import binding as B
from speculative_decoding_tree_parent_gb300 import workloads as W
from speculative_decoding_tree_parent_gb300.step import DeviceBatch

import attn_tolerance as AT

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)

def _both(inp):
    sep = DeviceBatch(inp)
    sep.build_mask()
    sep.attention()
    fused = DeviceBatch(inp)
    fused.out.fill_(float("nan"))
    fused.attention_parents()
    torch.cuda.synchronize()
    assert sep.device_status() == 0 and fused.device_status() == 0
    return sep, fused


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_fused_mask_equals_mask_then_attention(cfg):
    inp = W.generate_index(cfg)
    sep, fused = _both(inp)
    assert torch.equal(sep.out, fused.out)
    assert torch.equal(sep.lse, fused.lse)


@pytest.mark.parametrize("prefix,nodes,tree,hq", [(1000, 256, "random", 32), (300, 200, "chain", 32),
                                                  (17, 5, "random", 32), (0, 64, "random", 32),
                                                  (4099, 130, "random", 64), (64 * 9, 1, "random", 8)])
def test_fused_mask_trees_and_shapes(prefix, nodes, tree, hq):
    """Trees over several 64-key blocks (256 nodes), a 199-deep chain, one node, no prefix,
    GQA groups of 1 to 8; compared with the two-call path and with the oracle."""
    sp = W.spec(3, batch=3, prefix=(max(0, prefix - 40), prefix), nodes=(nodes, nodes) if tree != "chain" else
                (nodes - 1, nodes - 1), hq=hq, vocab=64, tree=tree, agree_prob=0.5,
                max_depth=nodes if tree == "chain" else 8)
    inp = W.generate(sp, seed=prefix + nodes)
    sep, fused = _both(inp)
    assert torch.equal(sep.out, fused.out)
    mask, _ = oracle.ancestor_mask_batch(inp.parent, inp.qo_indptr, inp.max_nodes)
    ref, _, A = AT.reference(inp, mask)
    AT.check(fused.out.float().cpu().numpy(), ref, A, "attention with the mask inside")


def test_fused_mask_reports_a_bad_parent():
    inp = W.generate_index(2)
    db = DeviceBatch(inp)
    par = db.parent.clone()
    par[10] = 10          # a node that is its own parent
    db.parent = par
    db.attention_parents()
    torch.cuda.synchronize()
    assert db.device_status() == -2


def test_fused_mask_refuses_unsupported_shapes():
    inp = W.generate_index(1)   # fp32, head dim 64: no tensor-core path
    db = DeviceBatch(inp)
    with pytest.raises(ValueError):
        db.attention_parents()  # the binding wants bf16 q
    lib = B.load()
    st = lib.spec_tree_verify_attn_parents(db.q.data_ptr(), db.k_pool.data_ptr(), db.v_pool.data_ptr(),
                                           db.k_pool.shape[0], 16, db.page_table.data_ptr(), db.page_table.shape[1],
                                           db.prefix_len.data_ptr(), db.max_prefix, db.k_tree.data_ptr(),
                                           db.v_tree.data_ptr(), db.parent.data_ptr(), db.qo.data_ptr(), 1, db.T,
                                           db.max_nodes, inp.hq, inp.hkv, inp.d, 0.0, db.out.data_ptr(), None,
                                           db.attn_ws.data_ptr(), db.attn_ws.numel(), None, None)
    assert st == -6
