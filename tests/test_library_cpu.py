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
