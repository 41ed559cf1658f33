"""Oracle: acceptance of the longest path of a draft tree, plus the bonus token.

Greedy ("EAGLE-2 deep dive", architecture section: the draft head's next token is
the argmax of the LM head; the target's logits are contrasted with the draft
tokens and the longest accepted path is fixed. "Accelerating Sonar through
speculation", speculative-decoding section: with n draft tokens up to n+1 tokens
come out, the extra one drawn from the target's logits at the mismatch or at the
end of the sequence):

  a[v] = argmax_t target_logits[v][t]         (reading: lowest token id on ties)
  v = root; repeat: take the first child c of v, in increasing node id, with
  draft_tokens[c] == a[v] (reading: among siblings with equal tokens the lowest
  id wins); stop when there is none. Bonus = a[stop node].

Stochastic ("EAGLE-2 deep dive", benchmark section: verification accepts or
rejects drafts by rejection sampling on the target's own distribution, lossless
at temperature 0 and under sampling; "Accelerating Sonar", draft-target section:
acceptance compares the complete draft and target distributions). The pages
give no formula; the reading taken is the standard speculative-sampling rule of
the works those pages cite (Leviathan et al.; Chen et al.), applied to the
children of a tree node one after another in the manner of SpecInfer's
multi-step tree verification (also cited there):

  p_v = softmax(target_logits[v] / T), q_v = softmax(draft_logits[v] / T)
  at node v start with r = p_v; for each child c of v in increasing id, x = token(c):
      accept c iff u_acc[c] < r(x) / q_v(x)   (q_v(x) == 0: accept iff r(x) > 0)
      on accept: move to c and repeat there
      on reject: r = max(r - q_v, 0) / sum(max(r - q_v, 0))   (sum 0: keep r)
  when no child is accepted (or v is a leaf): bonus = smallest t with
      sum_{t' <= t} r(t') > u_bonus[v] * sum_t r(t)     (inverse-CDF draw)

Near-ties: a ratio test with |u_acc - r(x)/q(x)| <= 1e-6, or a bonus draw whose
threshold u_bonus * sum(r) lies within 1e-8 * sum(r) of a CDF boundary, sets the
sequence's flag (bit 0 for a ratio test, bit 1 for the bonus draw); decisions
after a flagged one depend on it and are not comparable bit for bit. Reading for
the bonus band (the pages give none): a float32 evaluation of the residual carries
a few ulp (< 3e-7) of independent relative error per token, and factors common to
all tokens cancel between the cumulative sums and the total, so over a vocabulary
of up to 2^17 tokens the normalised cumulative sum is off by well under 1e-8; a
band of 1e-6 * sum(r) would instead flag about a quarter of all draws over 128K
nearly-uniform tokens, whose CDF steps are ~8e-6 apart.
"""

from dataclasses import dataclass

import numpy as np

TIE_EPS = 1e-6        # ratio tests: |u - r(x)/q(x)| <= TIE_EPS
BONUS_EPS = 1e-8      # bonus draw: |cdf boundary - u * sum(r)| <= BONUS_EPS * sum(r)
FLAG_RATIO = 1
FLAG_BONUS = 2


@dataclass
class AcceptResult:
    accept_len: np.ndarray   # int32 [B]  accepted draft nodes (root excluded)
    path: np.ndarray         # int32 [B, cap]  root + accepted nodes (sequence-local ids), -1 after
    out_tokens: np.ndarray   # int32 [B, cap]  accepted draft tokens then the bonus token, -1 after
    flags: np.ndarray        # uint8 [B]


def _children(parent_local, v):
    return [c for c in range(v + 1, len(parent_local)) if int(parent_local[c]) == v]


def _alloc(B, cap):
    return (np.zeros(B, np.int32), np.full((B, cap), -1, np.int32),
            np.full((B, cap), -1, np.int32), np.zeros(B, np.uint8))


def greedy_accept(parent, draft_tokens, target_logits, qo_indptr, path_cap):
    """Greedy longest accepted path + bonus token (see module docstring)."""
    qo = np.asarray(qo_indptr, np.int64)
    B = qo.shape[0] - 1
    acc, path, toks, flags = _alloc(B, path_cap)
    for b in range(B):
        a, e = int(qo[b]), int(qo[b + 1])
        if e == a:
            continue
        par = np.asarray(parent[a:e])
        tok = np.asarray(draft_tokens[a:e])
        v = 0
        nodes = [0]
        while True:
            best = int(np.argmax(target_logits[a + v]))  # first maximal index
            nxt = None
            for c in _children(par, v):
                if int(tok[c]) == best:
                    nxt = c
                    break
            if nxt is None:
                bonus = best
                break
            v = nxt
            nodes.append(v)
        L = len(nodes) - 1
        if L + 1 > path_cap:
            raise ValueError("path_cap too small for the accepted path")
        acc[b] = L
        path[b, : L + 1] = nodes
        toks[b, :L] = [int(tok[c]) for c in nodes[1:]]
        toks[b, L] = bonus
    return AcceptResult(acc, path, toks, flags)


def _softmax(x, temperature):
    z = np.asarray(x, np.float64) / float(temperature)
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def stochastic_accept(parent, draft_tokens, target_logits, draft_logits, uniforms,
                      temperature, qo_indptr, path_cap):
    """Speculative rejection sampling along the tree + residual bonus draw (module docstring)."""
    if not temperature > 0:
        raise ValueError("stochastic acceptance needs temperature > 0")
    qo = np.asarray(qo_indptr, np.int64)
    B = qo.shape[0] - 1
    acc, path, toks, flags = _alloc(B, path_cap)
    for b in range(B):
        a, e = int(qo[b]), int(qo[b + 1])
        if e == a:
            continue
        par = np.asarray(parent[a:e])
        tok = np.asarray(draft_tokens[a:e])
        v = 0
        nodes = [0]
        flag = 0
        while True:
            p = _softmax(target_logits[a + v], temperature)
            q = _softmax(draft_logits[a + v], temperature)
            r = p
            nxt = None
            for c in _children(par, v):
                x = int(tok[c])
                u = float(uniforms[a + c][0])
                if q[x] > 0:
                    ratio = r[x] / q[x]
                    if abs(u - ratio) <= TIE_EPS:
                        flag |= FLAG_RATIO
                    ok = u < ratio
                else:
                    ok = r[x] > 0
                if ok:
                    nxt = c
                    break
                res = np.maximum(r - q, 0.0)
                s = res.sum()
                if s > 0:
                    r = res / s
            if nxt is None:
                u = float(uniforms[a + v][1])
                cdf = np.cumsum(r)
                total = cdf[-1]
                thr = u * total
                t = int(np.searchsorted(cdf, thr, side="right"))
                t = min(t, len(r) - 1)
                lo = cdf[t - 1] if t > 0 else 0.0
                if abs(cdf[t] - thr) <= BONUS_EPS * total or (t > 0 and abs(lo - thr) <= BONUS_EPS * total):
                    flag |= FLAG_BONUS
                bonus = t
                break
            v = nxt
            nodes.append(v)
        L = len(nodes) - 1
        if L + 1 > path_cap:
            raise ValueError("path_cap too small for the accepted path")
        acc[b] = L
        path[b, : L + 1] = nodes
        toks[b, :L] = [int(tok[c]) for c in nodes[1:]]
        toks[b, L] = bonus
        flags[b] = flag
    return AcceptResult(acc, path, toks, flags)
