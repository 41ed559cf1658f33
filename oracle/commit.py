"""Oracle: commit of the accepted path's K/V into the sequence's paged cache.

"EAGLE-2 deep dive", architecture section: verifying the tree must not
contaminate the target model's KV cache. "Accelerating Sonar through
speculation": the KV entries of accepted tokens are filled before the next
decode step (draft-target section) and, in the MTP schedule, a kernel places
the next token after the shift with no CPU-GPU sync.

Reading (pages silent on the exact move): the tree's K/V arrive in a dense
buffer [T, Hkv, D] separate from the cache; the root (the last accepted token,
not yet in the verified prefix) and the L accepted nodes are written, in path
order, to logical slots P_b .. P_b + L of sequence b through its page table; the
new sequence length is P_b + L + 1. The bonus token's K/V does not exist yet (it
is the next step's root), so nothing is written for it. Every other byte of the
pool is left as it was.
"""

import numpy as np

from .fp8 import kv_quantize


def kv_commit(k_pool, v_pool, page_table, prefix_len, k_tree, v_tree, path, accept_len,
              qo_indptr, page_size=16, kv_scale=None):
    """Returns (new k_pool, new v_pool, seq_len int32 [B]); the inputs are not modified.

    With `kv_scale` [2, Hkv] the pools hold E4M3 codes: a committed row of KV head g is
    written as the codes of k_tree / kv_scale[0][g] (and v_tree / kv_scale[1][g]), the
    division in fp32 (oracle.fp8.kv_quantize)."""
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    qo = np.asarray(qo_indptr, np.int64)
    B = qo.shape[0] - 1
    seq_len = np.zeros(B, np.int32)
    for b in range(B):
        P = int(prefix_len[b])
        L = int(accept_len[b])
        a = int(qo[b])
        for i in range(L + 1):
            node = int(path[b][i])
            slot = P + i
            page = int(page_table[b][slot // page_size])
            if page < 0 or page >= kp.shape[0]:
                raise ValueError("no cache page for a committed slot")
            if kv_scale is None:
                kp[page, :, slot % page_size, :] = k_tree[a + node]
                vp[page, :, slot % page_size, :] = v_tree[a + node]
            else:
                kp[page, :, slot % page_size, :] = kv_quantize(k_tree[a + node], np.asarray(kv_scale[0])[:, None])
                vp[page, :, slot % page_size, :] = kv_quantize(v_tree[a + node], np.asarray(kv_scale[1])[:, None])
        seq_len[b] = P + L + 1
    return kp, vp, seq_len


def token_insert(token_buf, prefix_len, out_tokens, accept_len):
    """The next step's tokens on the device ("Accelerating Sonar", MTP-schedule section: a
    kernel places the next token after the shift, with no CPU-GPU sync).

    Reading (the page gives the idea, not the layout): row b of token_buf holds sequence b's
    tokens by position, its root (the last accepted token) at P_b; the step appends its L_b
    accepted tokens and then the bonus token, in that order, at positions P_b + 1 ..
    P_b + L_b + 1 -- the bonus is the root of the next step, at the new sequence length.
    Returns the new buffer; the input is not modified. A row too short raises."""
    buf = np.array(token_buf, copy=True)
    for b in range(buf.shape[0]):
        P, L = int(prefix_len[b]), int(accept_len[b])
        if P + L + 1 >= buf.shape[1]:
            raise ValueError("token row too short for the step's tokens")
        for i in range(L + 1):
            buf[b, P + 1 + i] = out_tokens[b][i]
    return buf
