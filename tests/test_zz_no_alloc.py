"""spec_accept_noalloc: acceptance for callers that cannot allocate device memory.

A caller such as a plugin host without an allocator, or a serving loop that forbids
allocation while it runs, has no workspace to pass. The library then uses a fixed
array of its own as scratch. This file checks, through the C ABI, that the
allocation-free entry point gives exactly what spec_accept gives with a caller
workspace, on two calls in a row (the second call finds the first call's leftovers in
the shared array), and that sizes beyond the fixed array are refused. It is named to
be collected last.
"""

import numpy as np
import pytest
import torch

from speculative_decoding_tree_parent_gb300 import binding as B
from speculative_decoding_tree_parent_gb300 import workloads as W
from speculative_decoding_tree_parent_gb300.step import DeviceBatch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


def _outputs(db):
    return (db.accept_len.cpu().numpy().copy(), db.path.cpu().numpy().copy(),
            db.out_tokens.cpu().numpy().copy(), db.flags.cpu().numpy().copy())


def _noalloc(db, mode):
    m = B.SPEC_STOCHASTIC if mode == "stochastic" else B.SPEC_GREEDY
    for t in (db.accept_len, db.path, db.out_tokens, db.flags):
        t.fill_(-7 if t.dtype != torch.uint8 else 99)   # poison: every output must be rewritten
    B.spec_accept_noalloc(m, db.parent, db.tokens, db.target_logits, db.qo, db.max_nodes, db.accept_len,
                          db.path, db.out_tokens, draft_logits=db.draft_logits if m else None,
                          uniforms=db.uniforms if m else None, temperature=db.inp.temperature, flags=db.flags,
                          dev_status=db.status)
    torch.cuda.synchronize()
    return _outputs(db)


@pytest.mark.parametrize("case", ["greedy-llama3-8b", "stochastic-small", "greedy-chains"])
def test_noalloc_matches_workspace_entry_point(case):
    if case == "greedy-llama3-8b":
        inp, mode = W.generate_index(2), "greedy"
    elif case == "stochastic-small":
        inp, mode = W.generate(W.spec(4, batch=3, prefix=(64, 64), nodes=(40, 40), vocab=20000, hq=8)), "stochastic"
    else:
        inp, mode = W.generate(W.spec(5, batch=24, prefix=(32, 64), vocab=3001)), "greedy"
    db = DeviceBatch(inp, mode=mode)
    db.accept(mode)
    torch.cuda.synchronize()
    want = _outputs(db)
    assert int(db.status.item()) == 0
    for call in range(2):
        got = _noalloc(db, mode)
        assert int(db.status.item()) == 0, call
        for g, w, name in zip(got, want, ("accept_len", "path", "out_tokens", "flags")):
            assert np.array_equal(g, w), (call, name)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    # 16384 nodes of 128256-token logits need more scratch than the fixed 4 MiB: the call is
    # refused on the host before anything is read, so small stand-in buffers suffice here
    T, V = 16384, 128256
    need = B.spec_workspace_size(B.SPEC_OP_ACCEPT, 1, T, 1024, 0, 0, 0, 0, V)
    assert need > (4 << 20)
    small = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = small.data_ptr()
    lib = B.load()
    st = lib.spec_accept_noalloc(B.SPEC_GREEDY, p, p, p, None, None, 1.0, V, p, 1, T, 1024, 9, p, p, p, None, None,
                                 None)
    assert st == -5
    torch.cuda.synchronize()
    assert int(small.abs().sum().item()) == 0   # nothing was written
