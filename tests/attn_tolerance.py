"""Per-element error bound of the bf16 tree-verify attention against the fp64 oracle.

bf16 keeps 8 significant bits, so rounding a value to bf16 (to nearest) moves it by at
most 2^-8 of itself. The tensor-core kernel's arithmetic, and what each step can add to an
output element (p_k = the exact softmax weights of the row, A = sum_k p_k |v_k|, o = the
exact output):
- scores and the O accumulator are fp32; P = exp2(score - running max) is rounded to bf16
  before the PV product, while the row sum adds the unrounded values: at most 2^-8 A;
- with key splits, each split's O / l is rounded to bf16 before the log-sum-exp merge.
  The merge is a convex combination whose weights times each split's own softmax weights
  are the p_k, so this adds at most 2^-8 A;
- the output is rounded to bf16: at most 2^-8 |o|;
- fp32 accumulation, ex2.approx and the rescale factors add terms far below 2^-16 A; the
  2^-12 A term covers them with room to spare.
So |gpu - oracle| <= (2^-7 + 2^-12) A + 2^-8 |o| element by element. A comes from the
oracle itself: the same attention with every value replaced by its absolute value. With
an FP8 cache the values are the codes' dequantised values (the widening to bf16 is exact
and the scales enter P's exponent and the row sum, not the operands), so the same bound
holds with A over the dequantised |v|.

This bound is tight enough to fail on a zeroed output and on an output that misses one key
split's share of the prefix (the negative controls below), unlike a bound scaled by the
largest |v|, which near-uniform softmax over thousands of keys can put above the outputs.
"""

from dataclasses import replace

import numpy as np

import oracle

P_REL = 2.0 ** -7 + 2.0 ** -12
O_REL = 2.0 ** -8
ABS = 1e-7
OUTER = 2e-2  # the stated max-abs-error bar for bf16 inputs, kept alongside


def _abs_values(v_pool, fp8):
    # E4M3 codes carry the sign in the top bit: clearing it gives the code of |value|
    return (np.asarray(v_pool) & np.uint8(0x7F)) if fp8 else np.abs(v_pool)


def reference(inp, mask, rows=None, pools=None, kv_scale=None, prefix_len=None):
    """(ref, lse, A): the oracle's output and lse for every row (rows=None) or for the
    sampled (node, head) rows, and the same attention over absolute values.
    pools: (k_pool, v_pool) in place of the input's (E4M3 codes when kv_scale is given);
    prefix_len: in place of the input's (the negative control shortens it)."""
    kp, vp = pools if pools is not None else (inp.k_pool, inp.v_pool)
    fp8 = kv_scale is not None
    P = inp.prefix_len if prefix_len is None else prefix_len
    vabs, vtabs = _abs_values(vp, fp8), np.abs(inp.v_tree)
    if rows is None:
        f = lambda v, vt: oracle.tree_verify_attention(inp.q, kp, v, inp.page_table, P, inp.k_tree, vt, mask,
                                                       inp.qo_indptr, inp.hq, inp.hkv, kv_scale=kv_scale)
    else:
        f = lambda v, vt: oracle.tree_verify_attention_rows(rows, inp.q, kp, v, inp.page_table, P, inp.k_tree, vt,
                                                            mask, inp.qo_indptr, inp.hq, inp.hkv, kv_scale=kv_scale)
    ref, lse = f(vp, inp.v_tree)
    A, _ = f(vabs, vtabs)
    return ref, lse, A


def bound(ref, A):
    return P_REL * A + O_REL * np.abs(ref) + ABS


def check(got, ref, A, what=""):
    """Assert the bound element by element (and the outer bar); returns the max error."""
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    tol = bound(ref, A)
    worst = int(np.argmax(err - tol))
    assert err.flat[worst] <= tol.flat[worst], (what, float(err.flat[worst]), float(tol.flat[worst]))
    assert err.max() <= OUTER, (what, float(err.max()))
    return float(err.max())


def rejects(wrong, ref, A):
    """Whether the bound rejects `wrong` (some element beyond it)."""
    return bool((np.abs(np.asarray(wrong, np.float64) - ref) > bound(ref, A)).any())


def negative_controls(inp, mask, ref, A, splits, rows=None, pools=None, kv_scale=None):
    """The check must reject (1) a zeroed output and (2) the output of the same attention
    without one key split's share of the prefix (each sequence's last ceil(P / S) prefix
    keys dropped; a quarter of them when the keys are not split). Both are made on the host
    from the oracle; nothing runs on the GPU."""
    assert rejects(np.zeros_like(ref), ref, A), "a zeroed output passes the bound"
    P = np.asarray(inp.prefix_len, np.int64)
    if P.max() == 0:
        return
    div = splits if splits > 1 else 4
    share = -(-P // div)
    short = np.maximum(P - share, 0).astype(np.int32)
    dropped, _, _ = reference(inp, mask, rows=rows, pools=pools, kv_scale=kv_scale, prefix_len=short)
    assert rejects(dropped, ref, A), "an output missing one split's keys passes the bound"


def with_q_scaled(inp, factor):
    """The inputs with q multiplied by a power of two (exact in bf16): a more peaked softmax."""
    return replace(inp, q=(inp.q * np.float32(factor)).astype(np.float32))
