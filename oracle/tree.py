"""Plain float64 oracle of tree drafting and tree verification.

TEST INFRASTRUCTURE, like spec_oracle.py: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import or run this module.

Source: "Speculative Decoding Part 1: 도입 전에 확인해야 할 것들" (VESSL AI blog),
section "gamma 재배분: 체인 대신 트리": draft a tree of candidate continuations
instead of one chain and verify it in one target pass (each branch sees only
its ancestors); choose the tree by scoring every node with its survival
probability a_v (the probability of reaching and accepting it) and taking the
global top-n -- a_v only decreases going down, so with ties broken towards the
shallower node the greedy choice is closed under prefixes and optimal for a
fixed budget.

Readings (the page gives no verification rule or data layout):
* Candidate tree: slots s = 0..N-1 of a request with parent[s] in {-1} or
  [0, s) (-1: the root, the anchor x_0); depth(s) = depth(parent) + 1, <= gamma.
  Each slot has a conditional survival factor c_s (supplied, e.g. from the
  confidence head); a_s is the fp32 product of the factors from the root down.
  Selection: top-n by a_s descending, ties by depth, then slot index.
* Drafting: a selected slot s at depth d + 1 with parent node p holds a token
  drawn from the Markov head's q_p = softmax((U_d + W1[x_p] W2) / T) with its
  own uniform (children of one node are independent draws from q_p).
* Verification, for independently drawn children (recursive rejection
  sampling, the multi-candidate form of the ratio test; it keeps the emitted
  sequence distributed as the target's): at node p with target p_p and draft
  q_p, try the selected children in slot order: child c is accepted iff
  u_accept[c] < r(x_c) / q_p(x_c), r starting at p_p; after a rejection r
  becomes normalize(max(0, r - q_p)) (kept if that has no mass).  An
  accepted child becomes the next node; if no child is accepted the final
  token is drawn from r with u_final (at a leaf, r = p_p: the bonus token).
* Target rows: target[b][0] at the root, target[b][1 + s] at slot s.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from oracle import spec_oracle as O


def depths(parent) -> np.ndarray:
    d = np.zeros(len(parent), np.int64)
    for s, p in enumerate(parent):
        assert p < s, "parents precede their children"
        d[s] = 1 if p < 0 else d[p] + 1
    return d


def survival(parent, conf32) -> np.ndarray:
    """a_s = c_s * a_parent in fp32 (root factor 1)."""
    c = np.asarray(conf32, dtype=np.float32)
    a = np.empty_like(c)
    for s, p in enumerate(parent):
        a[s] = c[s] if p < 0 else np.float32(a[p] * c[s])
    return a


def select(parent, conf32, n: int) -> np.ndarray:
    """Mask of the top-n slots by survival (ties: shallower, then lower index)."""
    a = survival(parent, conf32)
    d = depths(parent)
    order = sorted(range(len(parent)), key=lambda s: (-float(a[s]), int(d[s]), s))
    mask = np.zeros(len(parent), bool)
    mask[order[:n]] = True
    return mask


def children(parent, mask, node: int) -> list:
    """Selected children of `node` (-1: the root) in slot order."""
    return [s for s, p in enumerate(parent) if p == node and mask[s]]


def node_draft(U_b, W1, W2, anchor, tokens, parent, node, T):
    """q of a node's children: U row = the node's depth, factor = its token."""
    if node < 0:
        return O.draft_distribution(U_b[0], W1, W2, int(anchor), T)
    d = int(depths(parent)[node])
    return O.draft_distribution(U_b[d], W1, W2, int(tokens[node]), T)


@dataclasses.dataclass
class TreeDraft:
    tokens: np.ndarray     # int32 [N], -1 for unselected slots
    q_tok: np.ndarray      # float64 [N]
    dist: np.ndarray       # float64 [N] boundary distance of each draw (inf unselected)


def draft_request(U_b, W1, W2, anchor, T, parent, mask, u_draft_b) -> TreeDraft:
    N = len(parent)
    tokens = np.full(N, -1, np.int32)
    q_tok = np.full(N, np.nan)
    dist = np.full(N, np.inf)
    for node in [-1] + list(range(N)):
        if node >= 0 and not mask[node]:
            continue
        kids = children(parent, mask, node)
        if not kids:
            continue
        q, _ = node_draft(U_b, W1, W2, anchor, tokens, parent, node, T)
        for c in kids:
            dr = O.inverse_cdf(q, float(u_draft_b[c]))
            tokens[c] = dr.token
            q_tok[c] = q[dr.token]
            dist[c] = dr.dist
    return TreeDraft(tokens, q_tok, dist)


@dataclasses.dataclass
class TreeVerify:
    path: list             # accepted slots, root to the last accepted node
    out_tokens: np.ndarray  # int32 [depth_max + 1]: accepted tokens, final token, -1
    final: O.Draw
    dmin: float            # smallest distance of a consumed uniform to its boundary


def verify_request(t_b, U_b, W1, W2, anchor, T, parent, mask, tokens, u_accept_b, u_final,
                   gamma: int) -> TreeVerify:
    node, path, dmin = -1, [], np.inf
    while True:
        row = 0 if node < 0 else 1 + node
        p, _ = O.target_distribution(t_b[row], T)
        kids = children(parent, mask, node)
        r = p
        nxt = None
        if kids:
            q, _ = node_draft(U_b, W1, W2, anchor, tokens, parent, node, T)
            for c in kids:
                x = int(tokens[c])
                ratio = r[x] / q[x]
                u = float(u_accept_b[c])
                dmin = min(dmin, abs(u - ratio))
                if u < ratio:
                    nxt = c
                    break
                res = np.maximum(0.0, r - q)
                z = float(np.sum(res))
                if z > 0.0:
                    r = res / z
        if nxt is None:
            final = O.inverse_cdf(r, float(u_final))
            dmin = min(dmin, final.dist)
            out = np.full(gamma + 1, -1, np.int32)
            out[:len(path)] = [tokens[s] for s in path]
            out[len(path)] = final.token
            return TreeVerify(path, out, final, dmin)
        path.append(nxt)
        node = nxt
