"""Oracle: the EAGLE-2 dynamic draft tree (test infrastructure only).

"EAGLE-2 deep dive" (techknowgenie), section on the dynamic draft-tree algorithm: a node's
confidence is the product of the draft probabilities along its path from the root; the
root's top-k children start a priority queue; the candidate with the highest confidence is
taken out and becomes the next node; unless it is at the depth limit, the draft head runs on
it and its top-k tokens are queued with confidence = parent's x the token's probability
(the page's listing drops those at or below a threshold); construction stops when the node
budget is reached.

Readings: node ids are given in the order nodes leave the queue (so parent[i] < i, the
convention the mask and verification calls use); ties in confidence go to the candidate
queued first; ties among a row's logits go to the lower token id; the probabilities are
softmax(logits) in fp64. `row_of(u)` returns the draft logits row of node u (the draft model
is outside the path); with row_key="edge" it is called as row_of(parent, token) instead, the
node's parent id (-1 for the root) and its token -- what a draft model conditions on.
"""

import numpy as np


def topk_softmax(row, k):
    """Top-k tokens of softmax(row) (largest logit first, lower id on ties) and their fp64
    probabilities."""
    x = np.asarray(row, np.float64)
    p = np.exp(x - x.max())
    p /= p.sum()
    idx = np.lexsort((np.arange(x.shape[0]), -x))[:k]
    return idx, p[idx]


def best_first_tree(row_of, root_token, n_nodes, topk, max_depth, threshold=0.0, tie_rel=1e-6, row_key="node"):
    """Returns (parent int32 [n], token int32 [n], score float64 [n], tight bool) where n <=
    n_nodes (fewer when the queue runs dry); `tight`: some pop had its best two confidences
    within a relative `tie_rel` (a kernel computing in lower precision may order it either
    way). row_key: "node" (row_of(u)) or "edge" (row_of(parent[u], token[u]))."""
    assert row_key in ("node", "edge")
    parent, token, score, depth = [-1], [int(root_token)], [1.0], [0]
    queue = []          # [confidence, parent, token, alive] in push order
    tight = False

    def expand(u):
        row = row_of(u) if row_key == "node" else row_of(parent[u], token[u])
        toks, probs = topk_softmax(row, topk)
        for t, p in zip(toks.tolist(), probs.tolist()):
            c = score[u] * p
            if threshold > 0 and not c > threshold:
                continue
            queue.append([c, u, int(t), True])

    if n_nodes > 1:
        expand(0)
    while len(parent) < n_nodes:
        best, second = None, -1.0
        for i, q in enumerate(queue):
            if not q[3]:
                continue
            if best is None or q[0] > queue[best][0]:
                if best is not None:
                    second = max(second, queue[best][0])
                best = i
            else:
                second = max(second, q[0])
        if best is None:
            break
        c, par, tok, _ = queue[best]
        queue[best][3] = False
        if second >= 0 and c - second <= tie_rel * c:
            tight = True
        nid = len(parent)
        parent.append(par)
        token.append(tok)
        score.append(c)
        depth.append(depth[par] + 1)
        if depth[nid] < max_depth and len(parent) < n_nodes:
            expand(nid)
    return (np.asarray(parent, np.int32), np.asarray(token, np.int32), np.asarray(score, np.float64), tight)
