"""CPU-side checks of the C-ABI library: it builds for sm_103a, loads without a GPU,
exports every function include/spec_verify.h declares, and its host-only helpers
(status strings, workspace sizes, launch plan) answer. No kernel is launched."""

import ctypes
import os
import re

import pytest

from speculative_decoding_tree_parent_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", txt))
    return names


@pytest.fixture(scope="module")
def lib():
    return binding.load(build.build())


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert {"spec_build_tree_mask", "spec_tree_verify_attn", "spec_accept", "spec_kv_commit"} <= declared
    raw = ctypes.CDLL(build.lib_path())
    for name in sorted(declared):
        assert hasattr(raw, name), name
    assert set(binding.EXPORTS) == declared


def test_status_strings(lib):
    for code in range(-9, 1):
        s = binding.status_string(code)
        assert s and s != "unknown status"
    assert binding.status_string(5) == "unknown status"


def test_workspace_sizes(lib):
    # config-2 shapes: split partials need workspace; accept needs counters + partials
    a = binding.spec_workspace_size(binding.SPEC_OP_ATTN, 1, 64, 64, 32, 8, 128, 4096, 0)
    c = binding.spec_workspace_size(binding.SPEC_OP_ACCEPT, 1, 64, 64, 0, 0, 0, 0, 128256)
    assert a % 256 == 0 and c % 256 == 0 and c > 0
    assert binding.spec_workspace_size(binding.SPEC_OP_ATTN, 1, 64, 64, 30, 8, 128, 4096, 0) == 0  # hq % hkv
    assert binding.spec_workspace_size(binding.SPEC_OP_ACCEPT, -1, 64, 64, 0, 0, 0, 0, 10) == 0


def test_attn_plan(lib):
    splits, tc = binding.spec_attn_plan(binding.SPEC_F32, 1, 16, 4, 1, 64, 16, 128)
    assert splits >= 1 and tc == 0          # fp32 always runs on the CUDA cores
    with pytest.raises(binding.SpecError):
        binding.spec_attn_plan(binding.SPEC_BF16, 1, 16, 4, 1, 96, 16, 128)   # head dim 96
    with pytest.raises(binding.SpecError):
        binding.spec_attn_plan(binding.SPEC_BF16, 1, 2000, 4, 1, 128, 16, 128)  # > 1024 nodes


def test_host_argument_checks_of_the_newer_entry_points(lib):
    """Checks that return before any device work: sizes, null pointers, unsupported shapes.
    The pointers passed are never dereferenced (each call returns at its host check)."""
    fake = ctypes.c_void_p(256)  # a non-null address the calls below never touch
    # draft tree: top-k beyond 16, a zero depth, a node budget beyond 1024, a short state
    st = lib.spec_tree_expand(fake, 1000, 1000, 1000, 1, 8, 17, 4, 0.0, fake, 1 << 20, fake, fake, fake, fake,
                              None, None, None)
    assert st == -1
    st = lib.spec_tree_expand(fake, 1000, 1000, 1000, 1, 8, 4, 0, 0.0, fake, 1 << 20, fake, fake, fake, fake,
                              None, None, None)
    assert st == -1
    assert lib.spec_tree_init(fake, 1, 2000, fake, 1 << 20, fake, fake, fake, fake, None, None) == -1
    need = binding.spec_workspace_size(binding.SPEC_OP_TREE, 2, 0, 64, 0, 0, 0, 0, 0)
    assert need > 0
    assert lib.spec_tree_init(fake, 2, 64, fake, need - 1, fake, fake, fake, fake, None, None) == -5
    # FP8 commit: head dim not a multiple of 16, then a missing scale array
    args = lambda d, scale: (fake, fake, scale, fake, 9, fake, fake, fake, 4, 4, 16, fake, None, fake, fake, 1, 4,
                             8, d, None, None)
    assert lib.spec_kv_commit_kv8(*args(24, fake)) == -6
    assert lib.spec_kv_commit_kv8(*args(32, None)) == -1
    # attention forms: an empty batch is a no-op, a head count that the KV heads do not
    # divide is refused before anything else
    common = lambda hq, hkv: (fake, fake, fake, 4, 16, fake, 4, fake, 64, fake, fake, fake, fake, 1, 4, 4, hq, hkv,
                              128, 0.0, fake, None, None, 0, None, None)
    assert lib.spec_tree_verify_attn_parents(*common(30, 8)) == -1
    c = list(common(32, 8))
    c[13] = 0   # batch 0
    assert lib.spec_tree_verify_attn_parents(*c) in (0, -6)   # no work, or no tensor-core path on this host
    kv8 = (fake, fake, fake, fake) + common(30, 8)[3:]
    assert lib.spec_tree_verify_attn_kv8(*kv8) == -1


def test_bf16_head128_runs_on_tensor_cores_only(lib):
    """A bf16 call with head dim 128 never falls back to the CUDA-core kernel: the plan says
    tensor cores (even on a host with no driver), shapes the tensor-core kernel does not
    serve are refused, and so are unaligned tensors. The pointers passed are never
    dereferenced (each call returns at its host check)."""
    splits, tc = binding.spec_attn_plan(binding.SPEC_BF16, 1, 64, 32, 8, 128, 16, 4096)
    assert tc == 1 and splits >= 1
    for hq, hkv, ps in [(24, 8, 16), (32, 8, 8), (32, 8, 32)]:   # group of 3; pages of 8 and 32
        with pytest.raises(binding.SpecError) as ei:
            binding.spec_attn_plan(binding.SPEC_BF16, 1, 64, hq, hkv, 128, ps, 4096)
        assert ei.value.status == -6
    # fp32 and head dim 64 stay on the CUDA cores, page size 8 included
    assert binding.spec_attn_plan(binding.SPEC_F32, 1, 64, 32, 8, 128, 8, 4096)[1] == 0
    assert binding.spec_attn_plan(binding.SPEC_BF16, 1, 64, 24, 8, 64, 8, 4096)[1] == 0

    fake, odd = ctypes.c_void_p(4096), ctypes.c_void_p(4098)   # 16-byte aligned / not

    def call(q=fake, hq=32, hkv=8, ps=16):
        return lib.spec_tree_verify_attn(binding.SPEC_BF16, q, fake, fake, 300, ps, fake, 300, fake, 4096, fake,
                                         fake, fake, fake, 1, 64, 64, hq, hkv, 128, 0.0, fake, None, fake, 1 << 30,
                                         None, None)
    assert call(hq=24) == -6          # group of 3
    assert call(ps=8) == -6           # 8-token pages
    assert call(q=odd) == -1          # q not 16-byte aligned
    try:
        import torch
        gpu = torch.cuda.is_available()
    except Exception:
        gpu = False
    if not gpu:   # no driver here: the tensor-map encoder is missing, which is an error
        assert call() == -7


def test_batches_past_a_launch_grid_are_refused(lib):
    """Sizes whose grid would exceed a launch's y / z extent (65535) are refused on the host
    (SPEC_ERR_UNSUPPORTED) instead of failing at launch: the attention's batch x KV heads, the
    stochastic acceptance's and the draft tree's sequences. Every call returns at its host
    check; the pointers are never dereferenced."""
    fake = ctypes.c_void_p(256)
    with pytest.raises(binding.SpecError) as ei:
        binding.spec_attn_plan(binding.SPEC_BF16, 8192, 64, 32, 8, 128, 16, 4096)   # 65536 (sequence, head) pairs
    assert ei.value.status == -6
    assert binding.spec_attn_plan(binding.SPEC_BF16, 8191, 64, 32, 8, 128, 16, 4096)[1] == 1
    common = lambda batch: (fake, fake, fake, 4, 16, fake, 4, fake, 64, fake, fake, fake, fake, batch, batch, 4, 32,
                            8, 128, 0.0, fake, None, None, 0, None, None)
    assert lib.spec_tree_verify_attn_parents(*common(8192)) == -6
    assert lib.spec_tree_verify_attn(binding.SPEC_BF16, *common(8192)) == -6
    # stochastic acceptance: 65536 sequences; greedy has no such limit (it stops later, here at
    # the workspace check: 0 bytes given)
    acc = lambda mode: (mode, fake, fake, fake, fake, fake, ctypes.c_float(1.0), 1000, fake, 65536, 65536, 4, 4,
                        fake, fake, fake, None, fake, 0, None, None)
    assert lib.spec_accept(*acc(binding.SPEC_STOCHASTIC)) == -6
    assert lib.spec_accept(*acc(binding.SPEC_GREEDY)) == -5
    # draft tree
    assert lib.spec_tree_init(fake, 65536, 64, fake, 1 << 40, fake, fake, fake, fake, None, None) == -6
    st = lib.spec_tree_expand(fake, 1000, 1000, 1000, 65536, 64, 4, 4, 0.0, fake, 1 << 40, fake, fake, fake, fake,
                              None, None, None)
    assert st == -6
    st = lib.spec_tree_expand_multi(fake, 1000, 1000, 1000, 65536, 64, 8, 4, 4, 0.0, fake, 1 << 40, fake, fake,
                                    fake, fake, fake, fake, fake, None, None, None)
    assert st == -6


def test_accept_plan(lib):
    """The read plan of spec_accept (host model only, given an SM count): the single-sequence
    64-node verify streams every row; 32 sequences of 64 nodes walk; stochastic always walks;
    an odd vocabulary (no 16-byte rows) streams."""
    G, S = binding.SPEC_GREEDY, binding.SPEC_STOCHASTIC
    assert binding.spec_accept_plan(G, 1, 64, 128256, 9, 152) == 0
    assert binding.spec_accept_plan(G, 32, 2048, 128256, 9, 152) == 1
    assert binding.spec_accept_plan(G, 128, 704, 128256, 9, 152) == 0    # short chains: the stream
    assert binding.spec_accept_plan(G, 32, 2048, 128255, 9, 152) == 0
    assert binding.spec_accept_plan(S, 1, 64, 128256, 9, 152) == 1
    with pytest.raises(binding.SpecError):
        binding.spec_accept_plan(G, 4, 3, 1000, 9, 152)   # fewer nodes than sequences


def test_early_reads_switch(lib):
    """spec_set_early_reads is host state only: off by default, returns the previous
    setting, and the context manager restores it."""
    assert binding.spec_set_early_reads(0) == 0      # the default is off
    assert binding.spec_set_early_reads(5) == 0      # any non-zero turns it on
    assert binding.spec_set_early_reads(1) == 1
    assert binding.spec_set_early_reads(0) == 1
    with binding.early_reads(True):
        assert binding.spec_set_early_reads(1) == 1
    assert binding.spec_set_early_reads(0) == 0


def test_logits_marshalling_refuses_pageable_host_tensors():
    """The binding passes logits as device tensors or pinned host tensors only; a pageable
    host tensor is refused before the library is called (the library refuses it too, with
    SPEC_ERR_ARG, where a device can answer the pointer query)."""
    import torch

    assert binding._logits_ptr(None) is None
    with pytest.raises(ValueError):
        binding._logits_ptr(torch.zeros((4, 8), dtype=torch.float32))
    with pytest.raises(ValueError):
        binding._ptr(torch.zeros(4, dtype=torch.int32))   # every other argument: device only
