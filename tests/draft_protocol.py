"""Host model of the multi-row draft-tree call's request protocol (test helper).

The pages' construction ("EAGLE-2 deep dive", section on the dynamic draft-tree algorithm)
pops one candidate at a time and runs the draft head on it. spec_tree_expand_multi batches
it without changing the tree: a candidate's expansion depends only on its parent and token,
so each call lists the node awaiting its expansion plus the best queued candidates without a
row yet, the caller's draft model writes those rows, and the next call pops exactly as the
one-row construction would, expanding at once every popped node whose row it already has.

This model runs that protocol with the oracle's fp64 top-k softmax, so the CPU tests can
check that it builds the oracle's tree for every width, and the GPU tests can compare the
number of calls and the requests per call with the device's.
"""

from dataclasses import dataclass, field

import numpy as np

import oracle.draft_tree as DT


@dataclass
class ProtocolRun:
    parent: np.ndarray
    token: np.ndarray
    calls: int
    requests: list = field(default_factory=list)   # per call: [(parent, token), ...]


def multi_row_tree(row_of_edge, root_token, n_nodes, topk, max_depth, width, threshold=0.0):
    """row_of_edge(parent, token) -> the draft logits row of the node those define (parent
    -1: the root). Returns the tree, the number of calls and each call's request list."""
    parent, token, score, depth = [-1], [int(root_token)], [1.0], [0]
    queue = []   # dicts: c, parent, token, alive, result (None or (tokens, probs))
    run = ProtocolRun(None, None, 0, [])
    cur = 0 if n_nodes > 1 else -1
    requests = [("node", 0)] if cur == 0 else []

    def push(u, res):
        for t, p in zip(res[0].tolist(), res[1].tolist()):
            c = score[u] * p
            if threshold > 0 and not c > threshold:
                continue
            queue.append(dict(c=c, parent=u, token=int(t), alive=True, result=None))

    while requests:
        run.calls += 1
        listed = []
        cur_res = None
        for kind, i in requests:
            if kind == "node":
                listed.append((parent[i], token[i]))
                cur_res = DT.topk_softmax(row_of_edge(parent[i], token[i]), topk)
            else:
                q = queue[i]
                listed.append((q["parent"], q["token"]))
                q["result"] = DT.topk_softmax(row_of_edge(q["parent"], q["token"]), topk)
        run.requests.append(listed)
        node, res = cur, cur_res
        while True:
            push(node, res)
            stop = None
            while stop is None:
                alive = [i for i, q in enumerate(queue) if q["alive"]]
                if not alive:
                    cur, stop = -1, 1
                    break
                best = min(alive, key=lambda i: (-queue[i]["c"], i))
                q = queue[best]
                q["alive"] = False
                nid = len(parent)
                parent.append(q["parent"])
                token.append(q["token"])
                score.append(q["c"])
                depth.append(depth[q["parent"]] + 1)
                if depth[nid] < max_depth and len(parent) < n_nodes:
                    if q["result"] is not None:
                        node, res, stop = nid, q["result"], 0
                    else:
                        cur, stop = nid, 1
                elif len(parent) < n_nodes:
                    continue          # at the depth limit: the next candidate
                else:
                    cur, stop = -1, 1  # budget met
            if stop == 1:
                break
        if cur < 0:
            requests = []
        else:
            eligible = [i for i, q in enumerate(queue)
                        if q["alive"] and q["result"] is None and depth[q["parent"]] + 1 < max_depth]
            eligible.sort(key=lambda i: (-queue[i]["c"], i))
            requests = [("node", cur)] + [("cand", i) for i in eligible[: width - 1]]
    run.parent = np.asarray(parent, np.int32)
    run.token = np.asarray(token, np.int32)
    return run


class EdgeRows:
    """Seeded draft rows keyed by (sequence, parent, token): N(0, scale^2) logits, plus
    `bump` added to one token chosen by the key (a confident draft head) when bump > 0."""

    def __init__(self, seed, vocab, scale=2.0, bump=0.0):
        self.seed, self.vocab, self.scale, self.bump = seed, vocab, scale, bump
        self.cache = {}

    def row(self, b, parent, token):
        key = (b, int(parent), int(token))
        r = self.cache.get(key)
        if r is None:
            rng = np.random.default_rng([self.seed, b, int(parent) + 1, int(token)])
            r = (rng.standard_normal(self.vocab) * self.scale).astype(np.float32)
            if self.bump > 0:
                r[int(rng.integers(0, self.vocab))] += np.float32(self.bump)
            self.cache[key] = r
        return r

    def of(self, b):
        return lambda parent, token: self.row(b, parent, token)
