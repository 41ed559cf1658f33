"""Oracle: ancestor mask of a draft tree given as a parent array.

Follows "EAGLE-2 deep dive" (techknowgenie), core-implementation section, the
end of the dynamic-tree construction: for every node, start at the node and walk
parent links up to the root, marking each visited node id in that node's row of
the boolean tree mask. Nodes are numbered in creation order (the root is node 0
and a node is numbered after its parent), so parent[i] < i.
"""

import numpy as np


def _check_parent(parent: np.ndarray) -> None:
    n = parent.shape[0]
    if n == 0:
        return
    if int(parent[0]) != -1:
        raise ValueError("root (node 0) must have parent -1")
    for i in range(1, n):
        p = int(parent[i])
        if not (0 <= p < i):
            raise ValueError(f"node {i}: parent {p} is not an earlier node")


def ancestor_mask(parent) -> tuple:
    """Dense mask M[i][j] = True iff j is i or an ancestor of i; plus depth[i].

    parent: sequence-local parent array of one tree (root = -1).
    depth[i] is the number of parent links from i to the root (root depth 0).
    """
    parent = np.asarray(parent, dtype=np.int64)
    _check_parent(parent)
    n = parent.shape[0]
    M = np.zeros((n, n), dtype=bool)
    depth = np.zeros(n, dtype=np.int64)
    for i in range(n):
        cur = i
        steps = 0
        while cur >= 0:
            M[i, cur] = True
            cur = int(parent[cur])
            steps += 1
        depth[i] = steps - 1
    return M, depth


def ancestor_mask_batch(parent, qo_indptr, max_nodes=None) -> tuple:
    """Masks of a batch of trees, padded to max_nodes columns.

    Returns (mask bool [T, max_nodes], depth int64 [T]); row t of sequence b uses
    sequence-local column ids.
    """
    parent = np.asarray(parent, dtype=np.int64)
    qo = np.asarray(qo_indptr, dtype=np.int64)
    sizes = np.diff(qo)
    if max_nodes is None:
        max_nodes = int(sizes.max()) if sizes.size else 0
    T = int(qo[-1]) if qo.size else 0
    mask = np.zeros((T, max_nodes), dtype=bool)
    depth = np.zeros(T, dtype=np.int64)
    for b in range(qo.shape[0] - 1):
        a, e = int(qo[b]), int(qo[b + 1])
        if e == a:
            continue
        M, dep = ancestor_mask(parent[a:e])
        mask[a:e, : e - a] = M
        depth[a:e] = dep
    return mask, depth


def pack_mask_words(mask: np.ndarray, words: int) -> np.ndarray:
    """Bit-pack a boolean mask into uint64 words: bit (j & 63) of word (j >> 6) = mask[:, j]."""
    T, n = mask.shape
    if n > 64 * words:
        raise ValueError("mask wider than the words given")
    out = np.zeros((T, words), dtype=np.uint64)
    for j in range(n):
        out[:, j >> 6] |= mask[:, j].astype(np.uint64) << np.uint64(j & 63)
    return out
