"""One verification step on the device: the four C-ABI calls in order.

DeviceBatch holds a batch's inputs in device memory (uploaded once from a
workloads.VerifyInputs or pinned host copies), the outputs and the two
workspaces, and issues spec_build_tree_mask -> spec_tree_verify_attn ->
spec_accept -> spec_kv_commit on one stream. Nothing is computed in Python.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def _t(a, dtype, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


class DeviceBatch:
    """Device-resident buffers of one batch and the calls of one verification step."""

    def __init__(self, inp, device="cuda", mode=None, kv_fp8=False):
        """kv_fp8: hold the paged pool as E4M3 codes with per-KV-head scales
        (workloads.fp8_pool) and run the FP8-cache attention and commit calls."""
        self.inp = inp
        self.kv_fp8 = bool(kv_fp8)
        self.device = device
        fdt = torch.float32 if inp.dtype == "f32" else torch.bfloat16
        self.fdt = fdt
        self.mode = mode or inp.modes[0]
        dev = device
        self.qo = _t(inp.qo_indptr, torch.int32, dev)
        self.parent = _t(inp.parent, torch.int32, dev)
        self.tokens = _t(inp.draft_tokens, torch.int32, dev)
        self.q = _t(inp.q, fdt, dev)
        self.k_tree = _t(inp.k_tree, fdt, dev)
        self.v_tree = _t(inp.v_tree, fdt, dev)
        if self.kv_fp8:
            from .workloads import fp8_pool
            kc, vc, sc = fp8_pool(inp)
            self.k_pool = _t(kc, torch.uint8, dev)
            self.v_pool = _t(vc, torch.uint8, dev)
            self.kv_scale = _t(sc, torch.float32, dev)
            self.kv_codes = (kc, vc, sc)
        else:
            self.k_pool = _t(inp.k_pool, fdt, dev)
            self.v_pool = _t(inp.v_pool, fdt, dev)
            self.kv_scale = None
        self.page_table = _t(inp.page_table, torch.int32, dev)
        self.prefix_len = _t(inp.prefix_len, torch.int32, dev)
        self.target_logits = _t(inp.target_logits, torch.float32, dev)
        self.draft_logits = None if inp.draft_logits is None else _t(inp.draft_logits, torch.float32, dev)
        self.uniforms = None if inp.uniforms is None else _t(inp.uniforms, torch.float32, dev)
        T, Bn = inp.total_nodes, inp.batch
        self.T, self.B = T, Bn
        self.max_nodes = inp.max_nodes
        self.max_prefix = inp.max_prefix
        self.path_cap = inp.path_cap
        W = inp.mask_words
        self.mask = torch.zeros((T, W), dtype=torch.int64, device=dev)
        self.depth = torch.zeros(T, dtype=torch.int32, device=dev)
        self.out = torch.zeros((T, inp.hq, inp.d), dtype=fdt, device=dev)
        self.lse = torch.zeros((T, inp.hq), dtype=torch.float32, device=dev)
        self.accept_len = torch.zeros(Bn, dtype=torch.int32, device=dev)
        self.path = torch.zeros((Bn, self.path_cap), dtype=torch.int32, device=dev)
        self.out_tokens = torch.zeros((Bn, self.path_cap), dtype=torch.int32, device=dev)
        self.flags = torch.zeros(Bn, dtype=torch.uint8, device=dev)
        self.seq_len = torch.zeros(Bn, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        attn_ws = B.spec_workspace_size(B.SPEC_OP_ATTN, Bn, T, self.max_nodes, inp.hq, inp.hkv, inp.d,
                                        self.max_prefix, 0)
        acc_ws = B.spec_workspace_size(B.SPEC_OP_ACCEPT, Bn, T, self.max_nodes, 0, 0, 0, 0, inp.vocab)
        self.attn_ws = torch.zeros(max(attn_ws, 256), dtype=torch.uint8, device=dev)
        self.acc_ws = torch.zeros(max(acc_ws, 256), dtype=torch.uint8, device=dev)

    # --- one-copy transfers -------------------------------------------------------------
    STEP_INPUTS = ("q", "k_tree", "v_tree", "parent", "qo", "tokens", "page_table", "prefix_len")
    STEP_RESULTS = ("accept_len", "path", "out_tokens", "seq_len")

    def pack(self, names):
        """Re-home the named tensors as views of one device buffer (256-byte aligned slots)
        and return a pinned host buffer with the same layout, so that one copy moves them
        all. Call it before capturing a graph that uses them."""
        slots, off = [], 0
        for name in names:
            t = getattr(self, name)
            slots.append((name, off))
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        dev_buf = torch.empty(max(off, 256), dtype=torch.uint8, device=self.device)
        host_buf = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()
        for name, o in slots:
            t = getattr(self, name)
            n = t.numel() * t.element_size()
            view = dev_buf[o:o + n].view(t.dtype).view(t.shape)
            view.copy_(t)
            host_buf[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
            setattr(self, name, view)
        return dev_buf, host_buf

    # --- the four calls -------------------------------------------------------------
    def build_mask(self, stream=None):
        return B.spec_build_tree_mask(self.parent, self.qo, self.max_nodes, self.mask, self.depth, self.status,
                                      stream)

    def attention(self, stream=None, sm_scale=0.0):
        if self.kv_fp8:
            return B.spec_tree_verify_attn_kv8(self.q, self.k_pool, self.v_pool, self.kv_scale, self.page_table,
                                               self.prefix_len, self.max_prefix, self.k_tree, self.v_tree,
                                               self.mask, self.qo, self.max_nodes, self.out, self.lse, self.attn_ws,
                                               sm_scale, self.status, stream)
        return B.spec_tree_verify_attn(self.q, self.k_pool, self.v_pool, self.page_table, self.prefix_len,
                                       self.max_prefix, self.k_tree, self.v_tree, self.mask, self.qo,
                                       self.max_nodes, self.out, self.lse, self.attn_ws, sm_scale, self.status,
                                       stream)

    def attention_parents(self, stream=None, sm_scale=0.0):
        """The attention with the mask step inside it (ancestor bits from the parent array)."""
        return B.spec_tree_verify_attn_parents(self.q, self.k_pool, self.v_pool, self.page_table, self.prefix_len,
                                               self.max_prefix, self.k_tree, self.v_tree, self.parent, self.qo,
                                               self.max_nodes, self.out, self.lse, self.attn_ws, sm_scale,
                                               self.status, stream)

    def fused_mask_ok(self):
        """Whether the attention call can build the mask itself (tensor-core shapes, bf16 cache)."""
        return not self.kv_fp8 and self.inp.dtype == "bf16" and self.attn_plan()[1] == 1

    def accept(self, mode=None, stream=None):
        mode = mode or self.mode
        m = B.SPEC_STOCHASTIC if mode == "stochastic" else B.SPEC_GREEDY
        return B.spec_accept(m, self.parent, self.tokens, self.target_logits, self.qo, self.max_nodes,
                             self.accept_len, self.path, self.out_tokens, self.acc_ws,
                             draft_logits=self.draft_logits if m else None,
                             uniforms=self.uniforms if m else None, temperature=self.inp.temperature,
                             flags=self.flags, dev_status=self.status, stream=stream)

    def commit(self, stream=None):
        if self.kv_fp8:
            return B.spec_kv_commit_kv8(self.k_tree, self.v_tree, self.kv_scale, self.path, self.accept_len, self.qo,
                                        self.page_table, self.prefix_len, self.k_pool, self.v_pool, self.seq_len,
                                        self.status, stream)
        return B.spec_kv_commit(self.k_tree, self.v_tree, self.path, self.accept_len, self.qo, self.page_table,
                                self.prefix_len, self.k_pool, self.v_pool, self.seq_len, self.status, stream)

    def accept_commit(self, mode=None, stream=None):
        """spec_accept then spec_kv_commit, as the one fused call (two calls with an FP8 cache)."""
        mode = mode or self.mode
        if self.kv_fp8:
            self.accept(mode, stream)
            return self.commit(stream)
        m = B.SPEC_STOCHASTIC if mode == "stochastic" else B.SPEC_GREEDY
        return B.spec_accept_commit(m, self.parent, self.tokens, self.target_logits, self.qo, self.max_nodes,
                                    self.accept_len, self.path, self.out_tokens, self.acc_ws, self.k_tree,
                                    self.v_tree, self.page_table, self.prefix_len, self.k_pool, self.v_pool,
                                    seq_len_out=self.seq_len, draft_logits=self.draft_logits if m else None,
                                    uniforms=self.uniforms if m else None, temperature=self.inp.temperature,
                                    flags=self.flags, dev_status=self.status, stream=stream)

    def step(self, mode=None, stream=None, fused=True, fuse_mask=False):
        """One full verification step: mask, attention, then acceptance + KV commit (one fused
        call, or the two separate ones). fuse_mask: the attention call builds the mask itself
        (spec_tree_verify_attn_parents), where the shapes allow. Returns the number of kernel
        launches issued."""
        if fuse_mask and self.fused_mask_ok():
            self.attention_parents(stream)
        else:
            self.build_mask(stream)
            self.attention(stream)
        if fused:
            self.accept_commit(mode, stream)
        else:
            self.accept(mode, stream)
            self.commit(stream)
        return self.launches_per_step(mode, fused, fuse_mask)

    def launches_per_step(self, mode=None, fused=True, fuse_mask=False):
        """Kernel launches of one step: mask 1, attention 1 (+1 merge kernel when the keys are
        split), then accept 1 (greedy) or 2 (stochastic) and commit 1 -- except that the fused
        greedy call of up to 4 sequences commits inside its acceptance kernel (bf16 cache)."""
        mode = mode or self.mode
        splits, _ = self.attn_plan()
        attn = 2 if splits > 1 else 1
        acc = 2 if mode == "stochastic" else 1
        commit = 0 if (fused and mode != "stochastic" and self.B <= 4 and not self.kv_fp8) else 1
        mask = 0 if (fuse_mask and self.fused_mask_ok()) else 1
        return mask + attn + acc + commit

    def attn_plan(self):
        inp = self.inp
        dt = B.SPEC_F32 if inp.dtype == "f32" else B.SPEC_BF16
        return B.spec_attn_plan(dt, self.B, self.max_nodes, inp.hq, inp.hkv, inp.d, inp.page_size,
                                self.max_prefix)

    def device_status(self) -> int:
        return int(self.status.item())
