"""Pins of the oracle's KV commit: the logical cache of each sequence, read back through
its page table, is the old prefix followed by the accepted path's tree rows; every
other pool byte is unchanged; the new length is P + L + 1."""

import numpy as np

import oracle


def test_commit_logical_view_and_untouched_bytes():
    rng = np.random.default_rng(0)
    ps, hkv, d = 4, 2, 8
    P_list = [5, 0, 12, 7]
    n_list = [6, 3, 9, 1]
    B = len(P_list)
    need = [-(-(P + n) // ps) for P, n in zip(P_list, n_list)]
    total = sum(need) + 2
    ids = rng.permutation(total)
    pt = np.full((B, max(need)), -1, np.int64)
    off = 0
    for b in range(B):
        pt[b, : need[b]] = ids[off : off + need[b]]
        off += need[b]
    kp = rng.standard_normal((total, hkv, ps, d)).astype(np.float32)
    vp = rng.standard_normal((total, hkv, ps, d)).astype(np.float32)
    qo = np.concatenate([[0], np.cumsum(n_list)])
    kt = rng.standard_normal((qo[-1], hkv, d)).astype(np.float32)
    vt = rng.standard_normal((qo[-1], hkv, d)).astype(np.float32)
    paths = [[0, 2, 5], [0], [0, 1, 4, 8], [0]]
    acc = np.array([len(p) - 1 for p in paths])
    path = np.full((B, 9), -1)
    for b, p in enumerate(paths):
        path[b, : len(p)] = p
    k2, v2, seq_len = oracle.kv_commit(kp, vp, pt, P_list, kt, vt, path, acc, qo, page_size=ps)
    assert seq_len.tolist() == [P + L + 1 for P, L in zip(P_list, acc)]
    touched = np.zeros((total, ps), bool)
    for b in range(B):
        for s in range(seq_len[b]):
            page, row = pt[b, s // ps], s % ps
            if s < P_list[b]:
                assert np.array_equal(k2[page, :, row], kp[page, :, row])
            else:
                node = paths[b][s - P_list[b]]
                assert np.array_equal(k2[page, :, row], kt[qo[b] + node])
                assert np.array_equal(v2[page, :, row], vt[qo[b] + node])
                touched[page, row] = True
    by_slot = lambda a: a.transpose(0, 2, 1, 3)   # [page, row, Hkv, D]
    assert np.array_equal(by_slot(k2)[~touched], by_slot(kp)[~touched])
    assert np.array_equal(by_slot(v2)[~touched], by_slot(vp)[~touched])
    # the inputs themselves are not modified
    assert not np.shares_memory(k2, kp)


def test_token_insert_extends_each_sequence_by_its_emitted_tokens():
    """After a step, reading row b up to the new length + 1 gives the old tokens up to the
    root, then exactly the step's emitted tokens (accepted, then bonus): the sequence grows
    by L + 1 tokens, the root stays where it was, and nothing else of the row changes."""
    rng = np.random.default_rng(3)
    B, stride = 4, 40
    P = np.array([0, 7, 20, 33])
    L = np.array([0, 3, 8, 2])
    buf = rng.integers(0, 1000, (B, stride)).astype(np.int32)
    out = np.full((B, 9), -1, np.int32)
    emitted = []
    for b in range(B):
        toks = rng.integers(0, 1000, L[b] + 1)
        out[b, : L[b] + 1] = toks
        emitted.append(toks)
    new = oracle.token_insert(buf, P, out, L)
    for b in range(B):
        n = P[b] + L[b] + 1               # the new sequence length (KV slots 0 .. P + L)
        assert np.array_equal(new[b, : P[b] + 1], buf[b, : P[b] + 1])     # history and root
        assert np.array_equal(new[b, P[b] + 1 : n + 1], emitted[b])       # the step's tokens
        assert new[b, n] == emitted[b][-1]                                # next root = bonus
        assert np.array_equal(new[b, n + 1 :], buf[b, n + 1 :])           # the rest untouched
    assert not np.shares_memory(new, buf)


def test_token_insert_rejects_a_short_row():
    buf = np.zeros((1, 5), np.int32)
    try:
        oracle.token_insert(buf, [2], np.zeros((1, 9), np.int32), [2])   # needs positions 3 .. 5
    except ValueError:
        return
    raise AssertionError("a row without room must be refused")
