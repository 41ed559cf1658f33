"""Seeded synthetic inputs for tree-speculative-decoding verification.

This module only draws random numbers and lays them out in the buffers the
verification path consumes. It performs none of the verification arithmetic
(no ancestor masks, attention, acceptance or KV commit): the CUDA path and the
CPU oracle each do that on their own, from what is returned here.

Shapes follow the workloads of the pages on EAGLE / EAGLE-2 / EAGLE-3 tree
speculation:
  * draft trees of 16-128 nodes, depth <= 8, top-k 10, built best-first by the
    cumulative product of draft probabilities ("EAGLE-2 deep dive", section on
    the dynamic draft tree: C(u) = prod s(u_i), priority-queue expansion, node
    budget 64 or 128);
  * Llama-3-8B / 70B-shaped attention heads (32 or 64 query heads, 8 KV heads,
    head dim 128) over a paged KV cache with 16-token pages;
  * a 128256-token vocabulary for target and draft logits.
The draft model and target model themselves are not part of this build: their
outputs (logits, K/V rows, queries) are drawn from the stated distributions.

Layout conventions (all row-major, sequence-local tree node ids):
  qo_indptr     int32 [B+1]          node range of sequence b: [qo_indptr[b], qo_indptr[b+1])
  parent        int32 [T]            parent[root] = -1, 0 <= parent[i] < i otherwise
  draft_tokens  int32 [T]            token of each node; the root holds the last accepted token
  q             f32   [T, Hq, D]     (bf16-representable values when dtype == "bf16")
  k_tree/v_tree f32   [T, Hkv, D]
  k_pool/v_pool f32   [num_pages, Hkv, page_size, D]
  page_table    int32 [B, max_pages] (-1 marks an unused entry)
  prefix_len    int32 [B]
  target_logits f32   [T, V]
  draft_logits  f32   [T, V] or None
  uniforms      f32   [T, 2] or None (u_acc, u_bonus) in [0, 1)
"""

from __future__ import annotations

import heapq
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import numpy as np

PAGE_SIZE = 16
LLAMA3_VOCAB = 128256


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), returned as float32.

    Pure data preparation: every value the bf16 path receives is then exactly
    representable, so the GPU upload (float32 -> bfloat16) is lossless and the
    oracle sees the very same numbers.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    lsb = (bits >> 16) & np.uint32(1)
    rounded = (bits + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return rounded.view(np.float32)


@dataclass
class VerifyInputs:
    """One batch of verification inputs (see the module docstring for layouts)."""

    name: str
    dtype: str
    hq: int
    hkv: int
    d: int
    page_size: int
    vocab: int
    qo_indptr: np.ndarray
    parent: np.ndarray
    draft_tokens: np.ndarray
    q: np.ndarray
    k_tree: np.ndarray
    v_tree: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    page_table: np.ndarray
    prefix_len: np.ndarray
    target_logits: np.ndarray
    draft_logits: Optional[np.ndarray]
    uniforms: Optional[np.ndarray]
    temperature: float
    modes: tuple
    sm_scale: float
    max_depth: int
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.qo_indptr.shape[0] - 1)

    @property
    def total_nodes(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def nodes_per_seq(self) -> np.ndarray:
        return np.diff(self.qo_indptr)

    @property
    def max_nodes(self) -> int:
        return int(self.nodes_per_seq.max()) if self.batch else 0

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_prefix(self) -> int:
        return int(self.prefix_len.max()) if self.batch else 0

    @property
    def mask_words(self) -> int:
        return max(1, (self.max_nodes + 63) // 64)

    @property
    def path_cap(self) -> int:
        """Row length of path / out_tokens: deepest node depth + 1 (root + accepted nodes)."""
        return self.max_depth + 1


@dataclass(frozen=True)
class Spec:
    """Recipe for one synthetic workload."""

    name: str
    index: int                 # seeds: global = index, sequence b = 1000 * index + b
    dtype: str                 # "f32" | "bf16"
    batch: int
    hq: int
    hkv: int
    d: int
    vocab: int
    prefix: tuple              # (lo, hi) inclusive, uniform
    tree: str                  # "random" | "eagle2" | "chain"
    nodes: tuple               # random/eagle2: (n, n); chain: (lo, hi) draft tokens
    max_depth: int
    topk: int = 10
    draft_sigma: float = 2.0   # eagle2 draft-probability logits ~ N(0, sigma^2) (when no draft logits)
    qkv_scale: float = 1.0
    bump: Optional[tuple] = None         # (prob, amount): raise target logit of the first child's token
    agree_prob: Optional[float] = None   # random tree: draft token = argmax(parent target) with this prob
    draft_noise: Optional[float] = None  # draft_logits = target + N(0, noise^2); None = no draft logits
    page_layout: str = "shuffled"        # "identity" | "shuffled"
    extra_pages: int = 0                 # pool pages beyond what the sequences use
    modes: tuple = ("greedy",)
    temperature: float = 1.0


# The five workloads of the verification path. Index 1 is the tiny fp32 case the
# oracle finishes in well under a second; index 2 is the Llama-3-8B-shaped
# single-sequence verify the throughput is quoted on.
SPECS = {
    1: Spec(name="tiny-fp32", index=1, dtype="f32", batch=1, hq=4, hkv=1, d=64, vocab=1000,
            prefix=(128, 128), tree="random", nodes=(16, 16), max_depth=4,
            agree_prob=0.7, page_layout="identity", qkv_scale=1.0),
    2: Spec(name="llama3-8b-single", index=2, dtype="bf16", batch=1, hq=32, hkv=8, d=128,
            vocab=LLAMA3_VOCAB, prefix=(4096, 4096), tree="eagle2", nodes=(64, 64), max_depth=8,
            topk=10, draft_sigma=2.0, qkv_scale=1.0 / np.sqrt(128.0), bump=(0.8, 4.0)),
    3: Spec(name="llama3-8b-batch32", index=3, dtype="bf16", batch=32, hq=32, hkv=8, d=128,
            vocab=LLAMA3_VOCAB, prefix=(512, 8192), tree="eagle2", nodes=(64, 64), max_depth=8,
            topk=10, draft_sigma=2.0, qkv_scale=1.0 / np.sqrt(128.0), bump=(0.8, 4.0)),
    4: Spec(name="llama-70b-32k-stochastic", index=4, dtype="bf16", batch=8, hq=64, hkv=8, d=128,
            vocab=LLAMA3_VOCAB, prefix=(32768, 32768), tree="eagle2", nodes=(128, 128), max_depth=8,
            topk=10, qkv_scale=1.0 / np.sqrt(128.0), draft_noise=0.5, modes=("stochastic",)),
    5: Spec(name="chain-b128", index=5, dtype="bf16", batch=128, hq=32, hkv=8, d=128,
            vocab=LLAMA3_VOCAB, prefix=(256, 4096), tree="chain", nodes=(1, 8), max_depth=8,
            qkv_scale=1.0 / np.sqrt(128.0), bump=(0.8, 4.0), draft_noise=0.5,
            modes=("greedy", "stochastic")),
}


def spec(index: int, **overrides) -> Spec:
    """The workload recipe `index` (1..5), optionally with fields overridden (smaller tests)."""
    return replace(SPECS[index], **overrides)


def _random_tree(rng, n, max_depth):
    parent = np.full(n, -1, np.int64)
    depth = np.zeros(n, np.int64)
    for i in range(1, n):
        cands = np.flatnonzero(depth[:i] < max_depth)
        p = int(rng.choice(cands))
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def _topk_softmax(logits: np.ndarray, k: int):
    """Top-k tokens of softmax(logits) (descending) and their probabilities."""
    k = min(k, logits.shape[0])
    idx = np.argpartition(-logits, k - 1)[:k]
    idx = idx[np.lexsort((idx, -logits[idx].astype(np.float64)))]
    x = logits.astype(np.float64)
    m = x.max()
    z = np.exp(x - m).sum()
    return idx, np.exp(x[idx] - m) / z


def _best_first_tree(n_nodes, topk, max_depth, expand):
    """Best-first draft tree: pop the candidate with the highest cumulative product
    of draft probabilities, give it the next node id, expand it with its top-k
    children, until the node budget is reached.

    expand(node_id) returns (tokens, probs) of the draft distribution at that node.
    Returns parent (sequence-local) and token arrays in node-id order.
    """
    parent, depth, score, token = [-1], [0], [1.0], [None]
    heap, order = [], 0

    def push(node):
        nonlocal order
        toks, probs = expand(node)
        for t, p in zip(toks.tolist(), probs.tolist()):
            heapq.heappush(heap, (-(score[node] * p), order, node, int(t)))
            order += 1

    if n_nodes > 1:
        push(0)
    while heap and len(parent) < n_nodes:
        negc, _, par, tok = heapq.heappop(heap)
        nid = len(parent)
        parent.append(par)
        depth.append(depth[par] + 1)
        score.append(-negc)
        token.append(tok)
        if depth[nid] < max_depth and len(parent) < n_nodes:
            push(nid)
    return np.asarray(parent, np.int64), token, np.asarray(score)


def _tree_depths(parent):
    depth = np.zeros(len(parent), np.int64)
    for i in range(1, len(parent)):
        depth[i] = depth[parent[i]] + 1
    return depth


def generate(sp: Spec, seed: Optional[int] = None) -> VerifyInputs:
    """Draw one batch of inputs for recipe `sp`.

    Seeds: the global generator (pool values, page placement) uses `seed`
    (default: the recipe index); sequence b uses 1000 * seed + b for its prefix
    length, tree, tokens, logits, queries, tree K/V and uniforms.
    """
    base = sp.index if seed is None else int(seed)
    g = np.random.Generator(np.random.PCG64(base))
    B, V = sp.batch, sp.vocab
    ps = PAGE_SIZE

    seqs = []
    for b in range(B):
        r = np.random.Generator(np.random.PCG64(1000 * base + b))
        lo, hi = sp.prefix
        P = int(r.integers(lo, hi + 1))
        if sp.tree == "chain":
            n_draft = int(r.integers(sp.nodes[0], sp.nodes[1] + 1))
            n = n_draft + 1
        else:
            n = int(sp.nodes[0])
        seqs.append(dict(rng=r, P=P, n=n))

    # ---- trees, tokens and logits (per sequence) ---------------------------------
    parents, tokens, tgt_rows, dft_rows, unis, depths = [], [], [], [], [], []
    for s in seqs:
        r, n = s["rng"], s["n"]
        root_tok = int(r.integers(0, V))
        tgt = np.empty((n, V), np.float32)
        dft = np.empty((n, V), np.float32) if sp.draft_noise is not None else None
        made = np.zeros(n, bool)

        def make_rows(node):
            if not made[node]:
                tgt[node] = r.standard_normal(V, dtype=np.float32)
                if dft is not None:
                    dft[node] = tgt[node] + np.float32(sp.draft_noise) * r.standard_normal(V, dtype=np.float32)
                made[node] = True

        if sp.tree == "random":
            parent = _random_tree(r, n, sp.max_depth)
            for i in range(n):
                make_rows(i)
            tok = np.empty(n, np.int64)
            tok[0] = root_tok
            for i in range(1, n):
                if sp.agree_prob is not None and r.random() < sp.agree_prob:
                    tok[i] = int(np.argmax(tgt[parent[i]]))
                else:
                    tok[i] = int(r.integers(0, V))
        elif sp.tree == "eagle2":
            def expand(node):
                if dft is not None:
                    # the draft distribution of this node is the one acceptance compares against
                    make_rows(node)
                    return _topk_softmax(dft[node], sp.topk)
                logits = np.float32(sp.draft_sigma) * r.standard_normal(V, dtype=np.float32)
                return _topk_softmax(logits, sp.topk)

            parent, toklist, _ = _best_first_tree(n, sp.topk, sp.max_depth, expand)
            for i in range(n):
                make_rows(i)
            tok = np.asarray([root_tok] + toklist[1:], np.int64)
        elif sp.tree == "chain":
            parent = np.arange(-1, n - 1, dtype=np.int64)
            for i in range(n):
                make_rows(i)
            tok = np.empty(n, np.int64)
            tok[0] = root_tok
            for i in range(1, n):
                src = dft[i - 1] if dft is not None else tgt[i - 1]
                tok[i] = int(np.argmax(src))
        else:
            raise ValueError(sp.tree)

        if sp.bump is not None:
            prob, amount = sp.bump
            for v in range(n):
                kids = np.flatnonzero(parent == v)
                if kids.size and r.random() < prob:
                    first = int(kids.min())
                    tgt[v, tok[first]] += np.float32(amount)

        parents.append(parent)
        tokens.append(tok)
        tgt_rows.append(tgt)
        dft_rows.append(dft)
        depths.append(_tree_depths(parent))
        if "stochastic" in sp.modes:
            unis.append(r.random((n, 2), dtype=np.float32))

    n_per = np.asarray([s["n"] for s in seqs], np.int64)
    qo_indptr = np.zeros(B + 1, np.int32)
    qo_indptr[1:] = np.cumsum(n_per)
    T = int(qo_indptr[-1])
    max_depth = int(max(int(dd.max()) for dd in depths)) if B else 0

    # ---- queries and tree K/V (per sequence) -------------------------------------
    scale = np.float32(sp.qkv_scale)
    q = np.empty((T, sp.hq, sp.d), np.float32)
    kt = np.empty((T, sp.hkv, sp.d), np.float32)
    vt = np.empty((T, sp.hkv, sp.d), np.float32)
    for b, s in enumerate(seqs):
        r, a, e = s["rng"], qo_indptr[b], qo_indptr[b + 1]
        q[a:e] = r.standard_normal((e - a, sp.hq, sp.d), dtype=np.float32) * scale
        kt[a:e] = r.standard_normal((e - a, sp.hkv, sp.d), dtype=np.float32) * scale
        vt[a:e] = r.standard_normal((e - a, sp.hkv, sp.d), dtype=np.float32) * scale

    # ---- paged KV pool -------------------------------------------------------------
    # Each sequence owns enough pages for its prefix plus every slot a commit can
    # write (prefix + nodes), so the cache never runs out of room for an accepted path.
    need = [-(-(s["P"] + s["n"]) // ps) for s in seqs]
    total = int(sum(need)) + int(sp.extra_pages)
    ids = np.arange(total, dtype=np.int64)
    if sp.page_layout == "shuffled":
        ids = g.permutation(total)
    max_pages = max(need) if B else 0
    page_table = np.full((B, max(max_pages, 1)), -1, np.int32)
    off = 0
    for b in range(B):
        page_table[b, : need[b]] = ids[off : off + need[b]]
        off += need[b]
    k_pool = g.standard_normal((total, sp.hkv, ps, sp.d), dtype=np.float32) * scale
    v_pool = g.standard_normal((total, sp.hkv, ps, sp.d), dtype=np.float32) * scale

    if sp.dtype == "bf16":
        q, kt, vt = round_to_bf16(q), round_to_bf16(kt), round_to_bf16(vt)
        k_pool, v_pool = round_to_bf16(k_pool), round_to_bf16(v_pool)

    draft_logits = None
    if sp.draft_noise is not None:
        draft_logits = np.concatenate(dft_rows, axis=0) if B else np.zeros((0, V), np.float32)
    return VerifyInputs(
        name=sp.name,
        dtype=sp.dtype,
        hq=sp.hq,
        hkv=sp.hkv,
        d=sp.d,
        page_size=ps,
        vocab=V,
        qo_indptr=qo_indptr,
        parent=np.concatenate(parents).astype(np.int32) if B else np.zeros(0, np.int32),
        draft_tokens=np.concatenate(tokens).astype(np.int32) if B else np.zeros(0, np.int32),
        q=q,
        k_tree=kt,
        v_tree=vt,
        k_pool=k_pool,
        v_pool=v_pool,
        page_table=page_table,
        prefix_len=np.asarray([s["P"] for s in seqs], np.int32),
        target_logits=np.concatenate(tgt_rows, axis=0) if B else np.zeros((0, V), np.float32),
        draft_logits=draft_logits,
        uniforms=np.concatenate(unis, axis=0) if unis else None,
        temperature=float(sp.temperature),
        modes=tuple(sp.modes),
        sm_scale=float(1.0 / np.sqrt(sp.d)),
        max_depth=max(max_depth, 1),
        meta=dict(spec=sp, seed=base),
    )


def generate_index(index: int, seed: Optional[int] = None, **overrides) -> VerifyInputs:
    """Shorthand: generate(spec(index, **overrides), seed)."""
    return generate(spec(index, **overrides), seed)


def subset(inp: VerifyInputs, seqs: Sequence[int]) -> VerifyInputs:
    """The sub-batch made of sequences `seqs` (pool and page ids kept as they are)."""
    seqs = [int(s) for s in seqs]
    starts = inp.qo_indptr[:-1]
    ends = inp.qo_indptr[1:]
    rows = np.concatenate([np.arange(starts[s], ends[s]) for s in seqs]) if seqs else np.zeros(0, np.int64)
    n = np.asarray([ends[s] - starts[s] for s in seqs], np.int64)
    qo = np.zeros(len(seqs) + 1, np.int32)
    qo[1:] = np.cumsum(n)
    pick = lambda a: None if a is None else a[rows]
    return replace(
        inp,
        qo_indptr=qo,
        parent=inp.parent[rows],
        draft_tokens=inp.draft_tokens[rows],
        q=inp.q[rows],
        k_tree=inp.k_tree[rows],
        v_tree=inp.v_tree[rows],
        page_table=inp.page_table[seqs],
        prefix_len=inp.prefix_len[seqs],
        target_logits=inp.target_logits[rows],
        draft_logits=pick(inp.draft_logits),
        uniforms=pick(inp.uniforms),
    )


def fp8_pool(inp: VerifyInputs):
    """Input for the FP8-cache calls: (k_codes, v_codes, kv_scale) drawn from the workload's
    own pool. kv_scale float32 [2, Hkv] is each KV head's largest |value| / 448 (K, then V);
    the codes (uint8, the pool's shape) are torch's float8_e4m3fn cast of value / scale, a
    library routine used here only to lay out test data."""
    import torch

    scales = []
    codes = []
    for pool in (inp.k_pool, inp.v_pool):
        amax = np.abs(pool).max(axis=(0, 2, 3)).astype(np.float32)
        s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
        x = torch.from_numpy(np.ascontiguousarray(pool, np.float32) / s[None, :, None, None])
        codes.append(x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        scales.append(s)
    return codes[0], codes[1], np.stack(scales).astype(np.float32)
