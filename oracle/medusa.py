"""fp64 CPU oracle of one Medusa decode step (test infrastructure only).

Each function follows one step of the method in the order the pages give it:
heads -> per-head top-k -> candidate tree -> tree-masked attention ->
lm_head logits of every tree node -> typical acceptance and longest accepted
prefix -> KV rows of the accepted path written into the cache.

Where the pages leave a step open, the reading taken is stated in the
function's docstring under "Reading".
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


# ---------------------------------------------------------------------------
# Rounding point mirrored from the device path
# ---------------------------------------------------------------------------

def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value (ties to even), kept in fp64.

    bfloat16 keeps 8 significant bits, i.e. the top 7 of fp64's 52 fraction
    bits; the discarded 45 bits are rounded half-to-even on the bit pattern.
    (Normal range only; the step's values never approach bf16's limits.)
    """
    a = np.ascontiguousarray(a, dtype=np.float64)
    bits = a.view(np.uint64).copy()
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    bits = bits + np.uint64((1 << 44) - 1) + lsb
    bits &= ~np.uint64((1 << 45) - 1)
    return bits.view(np.float64)


# ---------------------------------------------------------------------------
# Heads  [ULT "How the heads predict the next tokens"; WIB "Medusa decoding heads"]
# ---------------------------------------------------------------------------

def medusa_heads(h: np.ndarray, W1: np.ndarray, b1: np.ndarray, W2: np.ndarray,
                 u_bf16: bool) -> Tuple[np.ndarray, np.ndarray]:
    """Medusa head k on hidden state h: logits_k = W2_k (h + SiLU(W1_k h + b1_k)).

    One fully connected layer with SiLU and a residual connection, then a
    bias-free projection onto the vocabulary [ULT]; every head reads the same
    last hidden state.  nn.Linear layout: W1 [K, H, H] and W2 [K, V, H] are
    [out, in].  Shapes: h [B, H] -> u [B, K, H], logits [B, K, V].

    Reading: the pages fix no precision.  The device path feeds u to the bf16
    W2 stream in bf16, so for bf16 workloads u is rounded to bf16 here too
    (u_bf16=True); fp32 workloads keep u unrounded.
    """
    h = np.asarray(h, np.float64)
    K = W1.shape[0]
    B = h.shape[0]
    u = np.empty((B, K, h.shape[1]))
    z = np.empty((B, K, W2.shape[1]))
    for k in range(K):
        a = h @ np.asarray(W1[k], np.float64).T + np.asarray(b1[k], np.float64)
        silu = a / (1.0 + np.exp(-a))                 # SiLU(a) = a * sigmoid(a)
        uk = h + silu
        if u_bf16:
            uk = bf16_round(uk)
        u[:, k] = uk
        z[:, k] = uk @ np.asarray(W2[k], np.float64).T
    return u, z


def tree_heads(X: np.ndarray, best_node: np.ndarray, W1: np.ndarray, b1: np.ndarray, W2: np.ndarray,
               u_bf16: bool) -> Tuple[np.ndarray, np.ndarray]:
    """The heads on the accepted node's hidden state, which the next step's
    candidates come from [WIB "Inference flow in an online chat service": the
    verification pass yields the next round's candidates with no extra pass;
    ULT "Tree attention and accepting tokens": the accepted branch continues].
    X [B, T, H] holds every tree node's state; row best_node[b] of request b
    goes through medusa_heads.  Returns (u, logits) as medusa_heads does.
    """
    X = np.asarray(X, np.float64)
    rows = X[np.arange(X.shape[0]), np.asarray(best_node)]
    return medusa_heads(rows, W1, b1, W2, u_bf16)


def head_topk(z: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Top-k candidates of each head's logits [WIB "Medusa decoding heads"; JIS].

    z [..., V] -> ids [..., k], vals [..., k], in descending value order.
    Reading: equal values are ordered by the lower token id (the pages do not
    say).  Also returns, per row, the decision margins: gaps between
    consecutive kept values and between the k-th kept and the best dropped
    value, used to recognise near-ties.
    """
    z = np.asarray(z, np.float64)
    V = z.shape[-1]
    flat = z.reshape(-1, V)
    ids = np.empty((flat.shape[0], k), np.int64)
    vals = np.empty((flat.shape[0], k))
    margin = np.empty(flat.shape[0])
    vid = np.arange(V)
    for r in range(flat.shape[0]):
        order = np.lexsort((vid, -flat[r]))          # primary: value desc, then id asc
        ids[r] = order[:k]
        vals[r] = flat[r, order[:k]]
        kept = flat[r, order[: min(k + 1, V)]]
        margin[r] = np.min(np.abs(np.diff(kept))) if kept.size > 1 else np.inf
    shp = z.shape[:-1]
    return ids.reshape(*shp, k), vals.reshape(*shp, k), margin.reshape(shp)


def base_root(h: np.ndarray, lm_head: np.ndarray) -> np.ndarray:
    """Root token on the first step: the base LM head's greedy next token.

    [ULT "How the heads predict the next tokens"]: the last hidden state at t
    goes to the language-model head, which scores token t+1; head k scores
    t+k+1.  [WIB "Typical acceptance"]: the first token is always taken
    greedily.  Reading: so the tree's root is argmax lm_head(h) (lowest id on
    ties) and depth d of the tree comes from head d.
    """
    z = np.asarray(h, np.float64) @ np.asarray(lm_head, np.float64).T
    return np.argmax(z, axis=-1)                     # numpy argmax returns the first maximum


# ---------------------------------------------------------------------------
# Candidate tree  [WIB "Tree attention"; ULT "Tree attention and accepting tokens"]
# ---------------------------------------------------------------------------

@dataclass
class TreeTables:
    nodes: List[Tuple[int, ...]]        # canonical order; nodes[0] == () is the root
    parent: np.ndarray                  # [T], -1 for the root
    depth: np.ndarray                   # [T]
    rank: np.ndarray                    # [T], rank within its head's top-k (-1 for root)
    ancestors: List[List[int]]          # ancestors(i) ordered root -> parent (excludes i)
    mask: np.ndarray                    # [T, T] bool, mask[i, j] = j is i or an ancestor of i
    leaves: List[int]                   # paths = root->leaf chains, leaves in canonical order
    children: List[List[int]]

    @property
    def T(self) -> int:
        return len(self.nodes)

    @property
    def dmax(self) -> int:
        return int(self.depth.max())


def tree_tables(choices: Sequence[Sequence[int]]) -> TreeTables:
    """Tables of a fixed candidate tree given as rank tuples ("medusa_choices").

    A choice (r1, ..., rd) is the node whose depth-j token is head j's rank-rj
    candidate; its parent is the tuple without its last rank.  Every branch
    at depth d takes head d's tokens, so the tree can be prepared once and its
    mask cached [WIB "Tree attention"; ULT].  Node order: root, then by depth,
    then by rank tuple.  A node may see only itself and its ancestors.
    Raises ValueError for a choice list that is not prefix-closed, has
    duplicates, empty tuples or negative ranks.
    """
    cs = [tuple(int(r) for r in c) for c in choices]
    if any(len(c) == 0 for c in cs):
        raise ValueError("empty choice")
    if any(r < 0 for c in cs for r in c):
        raise ValueError("negative rank")
    if len(set(cs)) != len(cs):
        raise ValueError("duplicate choice")
    s = set(cs)
    for c in cs:
        if len(c) > 1 and c[:-1] not in s:
            raise ValueError(f"choice {c} lacks its parent {c[:-1]}")
    nodes = [()] + sorted(cs, key=lambda t: (len(t), t))
    idx = {n: i for i, n in enumerate(nodes)}
    T = len(nodes)
    parent = np.full(T, -1, np.int64)
    depth = np.zeros(T, np.int64)
    rank = np.full(T, -1, np.int64)
    children: List[List[int]] = [[] for _ in range(T)]
    for i, n in enumerate(nodes[1:], start=1):
        parent[i] = idx[n[:-1]]
        depth[i] = len(n)
        rank[i] = n[-1]
        children[parent[i]].append(i)
    ancestors: List[List[int]] = []
    for i in range(T):
        chain = []
        p = parent[i]
        while p >= 0:
            chain.append(int(p))
            p = parent[p]
        ancestors.append(chain[::-1])
    mask = np.zeros((T, T), bool)
    for i in range(T):
        mask[i, i] = True
        mask[i, ancestors[i]] = True
    leaves = [i for i in range(T) if not children[i]]
    return TreeTables(nodes, parent, depth, rank, ancestors, mask, leaves, children)


def tree_tokens(tt: TreeTables, root: np.ndarray, topk_ids: np.ndarray,
                kv_len: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Token and position id of every tree node, per request.

    token(root) = root token; token(r1..rd) = head d's rank-rd candidate, the
    same head-d tokens under every branch [ULT "Tree attention and accepting
    tokens"].  Position = prefix length + depth [WIB "Tree attention": each
    token gets its correct position index].  Reading: the absolute position of
    a depth-d node is kv_len + d; depth alone is its offset from the prefix.
    topk_ids: [B, K, k] (head index 0 is head 1).
    """
    B = len(root)
    tok = np.empty((B, tt.T), np.int64)
    pos = np.empty((B, tt.T), np.int64)
    for b in range(B):
        for i, n in enumerate(tt.nodes):
            d = len(n)
            tok[b, i] = root[b] if d == 0 else topk_ids[b, d - 1, n[-1]]
            pos[b, i] = kv_len[b] + d
    return tok, pos


# ---------------------------------------------------------------------------
# Tree attention  [WIB "Tree attention"; ULT "Tree attention and accepting tokens"]
# ---------------------------------------------------------------------------

def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half form (Su et al., "RoFormer", 2021).

    x [..., n, D] with positions [...] (one position per leading index, shared by
    the n heads): for d < D/2, the pair (x[d], x[d + D/2]) is rotated by the angle
    position * theta^(-2d/D).  Used to make the tree's position ids matter
    [WIB "Tree attention": every candidate token gets its correct position index].
    """
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    half = D // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / D)
    ang = np.asarray(positions, np.float64)[..., None, None] * inv_freq      # [..., 1, D/2]
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def tree_attention(q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                   k_cache: np.ndarray, v_cache: np.ndarray, kv_len: np.ndarray,
                   tt: TreeTables, scale: float,
                   only: Optional[Sequence[Tuple[int, int, int]]] = None,
                   positions: Optional[np.ndarray] = None, rope_theta: float = 10000.0) -> np.ndarray:
    """One attention pass of all tree tokens over the KV cache plus the tree.

    Node i (query head hq) attends to the L = kv_len[b] cached keys and to
    the tree keys of its ancestors and itself, nothing else -- the tree mask
    [WIB "Tree attention"]: o = softmax(scale * q K^T) V over that key set.
    Shapes: q [B,T,Hq,D]; k_new, v_new [B,T,Hkv,D]; caches [B,Hkv,Lmax,D];
    returns o [B,T,Hq,D] (fp64).

    Reading: q/k/v are the layer's post-projection (post-RoPE) inputs, as the
    backbone that makes them is outside this step; query head hq uses key
    head floor(hq * Hkv / Hq) (grouped-query attention).  With ``positions``
    [B, T] given, the tree's q and k_new are first rotated at those positions
    (apply_rope); the cache keys are taken as already rotated at theirs.
    ``only`` limits the work to the listed (b, i, hq) outputs (others left NaN).
    """
    if positions is not None:
        q = apply_rope(q, positions, rope_theta)
        k_new = apply_rope(k_new, positions, rope_theta)
    B, T, Hq, D = q.shape
    Hkv = k_new.shape[2]
    out = np.full((B, T, Hq, D), np.nan)
    if only is None:
        only = [(b, i, hq) for b in range(B) for i in range(T) for hq in range(Hq)]
    for b, i, hq in only:
        g = hq * Hkv // Hq
        L = int(kv_len[b])
        sel = np.nonzero(tt.mask[i])[0]
        keys = np.concatenate([np.asarray(k_cache[b, g, :L], np.float64),
                               np.asarray(k_new[b, sel, g], np.float64)])
        vals = np.concatenate([np.asarray(v_cache[b, g, :L], np.float64),
                               np.asarray(v_new[b, sel, g], np.float64)])
        s = scale * (keys @ np.asarray(q[b, i, hq], np.float64))
        s = s - s.max()
        p = np.exp(s)
        p /= p.sum()
        out[b, i, hq] = p @ vals
    return out


# ---------------------------------------------------------------------------
# Verification logits and typical acceptance
# ---------------------------------------------------------------------------

def verify_logits(X: np.ndarray, lm_head: np.ndarray) -> np.ndarray:
    """lm_head logits of every tree node: z[b, i] = lm_head . X[b, i].

    The verification pass scores every candidate token of the tree in one go
    [WIB "Inference flow in an online chat service"]; X [B,T,H] holds the
    tree nodes' last hidden states (inputs here), lm_head is [V, H].
    """
    return np.asarray(X, np.float64) @ np.asarray(lm_head, np.float64).T


def node_posterior(z_parent: np.ndarray, token: int, temperature: float,
                   threshold: float, alpha: float) -> Dict[str, float]:
    """Typical-acceptance test of one candidate token given its parent's logits.

    temperature 0: accept iff the token is the model's greedy choice
    [ULT "Tree attention and accepting tokens"; WIB "Typical acceptance"].
    temperature > 0: q = softmax(z / temperature), p = q[token], entropy
    H = -sum q ln q; accept iff p > min(threshold, alpha * exp(-H)) -- the
    minimum of a hard threshold and an entropy-dependent one [WIB "Typical
    acceptance"], posterior_threshold 0.09 and posterior_alpha 0.3 [CNN].

    Reading: H is taken over the same temperature-scaled distribution as p,
    which is what makes the threshold fall as temperature rises [WIB "How the
    acceptance rate shapes the speedup"]; natural log; strict ">".  Greedy
    ties go to the lowest token id.  Returns p, H, the effective threshold,
    the decision and its margin (for near-tie accounting): |ln p - ln thr_eff|
    at temperature > 0, the top-1/top-2 logit gap at temperature 0.
    """
    z = np.asarray(z_parent, np.float64)
    top = int(np.argmax(z))
    srt = np.sort(z)
    gap = float(srt[-1] - srt[-2]) if z.size > 1 else np.inf
    if temperature == 0.0:
        return dict(p=float(token == top), H=0.0, thr=1.0, accept=bool(token == top),
                    margin=gap, argmax=top)
    y = z / temperature
    y = y - y.max()
    e = np.exp(y)
    S = e.sum()
    qv = e / S
    p = float(qv[token])
    nz = qv > 0
    H = float(-(qv[nz] * np.log(qv[nz])).sum())
    thr = min(threshold, alpha * np.exp(-H))
    margin = abs(np.log(p) - np.log(thr)) if p > 0 else np.inf
    return dict(p=p, H=H, thr=float(thr), accept=bool(p > thr), margin=float(margin), argmax=top)


def nucleus_next(z: np.ndarray, temperature: float, top_p: float, u: float) -> Dict[str, float]:
    """Next token drawn from the top-p nucleus of softmax(z / temperature), with the
    draw u in [0, 1) given [CNN "Posterior probability evaluation":
    evaluate_posterior(..., top_p=top_p, sampling=sampling) names nucleus sampling].

    Reading (the pages name the parameter only): the nucleus is the shortest run
    of tokens in descending probability, equal probabilities by the lower id,
    whose mass reaches top_p; the draw picks by inverse CDF over the nucleus
    renormalised, tokens in ascending id order (the first token whose running
    mass exceeds u times the nucleus mass).  Temperature 0 is the greedy token.
    Returns the token, the nucleus size and a margin for near-tie accounting
    (the smallest gap, relative to the nucleus mass, between u times the mass
    and a running-mass step, or between top_p and the mass at the nucleus edge).
    """
    z = np.asarray(z, np.float64)
    V = z.size
    if temperature == 0.0:
        srt = np.sort(z)
        return dict(token=int(np.argmax(z)), size=1, margin=float(srt[-1] - srt[-2]) if V > 1 else np.inf)
    y = (z - z.max()) / temperature
    q = np.exp(y)
    q /= q.sum()
    order = np.lexsort((np.arange(V), -q))
    cum = np.cumsum(q[order])
    n = min(V, int(np.searchsorted(cum, top_p, side="left")) + 1)
    members = np.sort(order[:n])
    mass = float(q[members].sum())
    target = u * mass
    run = np.cumsum(q[members])
    j = min(n - 1, int(np.searchsorted(run, target, side="right")))
    edge = [abs(cum[n - 1] - top_p)] + ([abs(cum[n - 2] - top_p)] if n >= 2 else [])
    margin = min(float(np.min(np.abs(run - target))) / mass, min(edge))
    return dict(token=int(members[j]), size=n, margin=margin)


def typical_accept(z: np.ndarray, tokens: np.ndarray, tt: TreeTables, temperature: float,
                   threshold: float, alpha: float, tie_break: str = "first") -> Dict[str, np.ndarray]:
    """Longest accepted prefix of the candidate tree, per request.

    A node is kept when its own token passes the acceptance test under its
    parent's logits and its parent is kept; the root (the greedy first token)
    is always kept [WIB "Typical acceptance"].  The longest kept branch wins
    [ULT "Tree attention and accepting tokens"]; its length is accept_length
    and its path is best_candidate [CNN "Posterior probability evaluation"].

    Reading: accept_length counts the tokens accepted beyond the root, i.e.
    the depth of the deepest kept node; among equally deep kept nodes the one
    first in canonical order wins (higher-ranked head candidates first), or,
    with tie_break="joint", the one whose path has the highest joint
    probability (the product of each node's p under its parent; the pages
    leave the choice open), equal products again to the first in canonical
    order;
    best_path is the first path (leaf in canonical order) through that node;
    the next root is the greedy token of the winner's logits [WIB "Inference
    flow": the next round starts from the last accepted token].
    z: [B, T, V] logits of every node; tokens: [B, T].
    """
    B, T = tokens.shape
    out = {k: [] for k in ("accept_len", "best_node", "best_path", "accepted_tokens",
                           "next_root", "node_p", "node_H", "node_accept", "margin", "joint_margin")}
    dmax = tt.dmax
    for b in range(B):
        p = np.full(T, np.nan)
        H = np.full(T, np.nan)
        acc_self = np.zeros(T, bool)
        margin = np.full(T, np.inf)
        for c in range(1, T):
            r = node_posterior(z[b, tt.parent[c]], int(tokens[b, c]), temperature, threshold, alpha)
            p[c], H[c], acc_self[c], margin[c] = r["p"], r["H"], r["accept"], r["margin"]
        kept = np.zeros(T, bool)
        kept[0] = True
        for c in range(1, T):                        # parents precede children in canonical order
            kept[c] = acc_self[c] and kept[tt.parent[c]]
        best = 0
        for c in range(1, T):
            if kept[c] and tt.depth[c] > tt.depth[best]:
                best = c
        joint_margin = np.inf
        if tie_break == "joint":
            # log joint probability of each kept node's path (root: ln 1 = 0)
            lp = np.zeros(T)
            for c in range(1, T):
                lp[c] = lp[tt.parent[c]] + (np.log(p[c]) if p[c] > 0 else -np.inf)
            deepest = [c for c in range(T) if kept[c] and tt.depth[c] == tt.depth[best]]
            best = max(deepest, key=lambda c: (lp[c], -c))
            others = [abs(lp[c] - lp[best]) for c in deepest if c != best]
            joint_margin = min(others) if others else np.inf
        elif tie_break != "first":
            raise ValueError(tie_break)
        a = int(tt.depth[best])
        chain = tt.ancestors[best] + [best]
        bp = next(pi for pi, leaf in enumerate(tt.leaves) if best == leaf or best in tt.ancestors[leaf])
        toks = np.full(dmax + 1, -1, np.int64)
        toks[: a + 1] = tokens[b, chain]
        out["accept_len"].append(a)
        out["best_node"].append(best)
        out["best_path"].append(bp)
        out["accepted_tokens"].append(toks)
        out["next_root"].append(int(np.argmax(z[b, best])))
        out["node_p"].append(p)
        out["node_H"].append(H)
        out["node_accept"].append(kept)
        out["margin"].append(margin)
        out["joint_margin"].append(joint_margin)
    return {k: np.array(v) for k, v in out.items()}


# ---------------------------------------------------------------------------
# KV commit  [WIB "Inference flow"; ULT "Tree attention and accepting tokens"]
# ---------------------------------------------------------------------------

def kv_commit(k_cache: np.ndarray, v_cache: np.ndarray, kv_len: np.ndarray,
              k_new: np.ndarray, v_new: np.ndarray, tt: TreeTables,
              best_node: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """Write the accepted path's tree K/V rows into the cache after the prefix.

    The kept branch continues the sequence [ULT]: the rows of its nodes
    root..best (depth 0..a) go to cache positions L..L+a and kv_len becomes
    L+a+1.  A request whose rows would pass the cache end (L+a+1 > Lmax) is
    left untouched and flagged (status 1).  Returns new caches, lengths and a
    per-request status.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    kl = np.array(kv_len, copy=True)
    status = np.zeros(len(kv_len), np.int64)
    Lmax = kc.shape[2]
    for b in range(len(kv_len)):
        chain = tt.ancestors[int(best_node[b])] + [int(best_node[b])]
        L = int(kv_len[b])
        if L + len(chain) > Lmax:
            status[b] = 1
            continue
        for d, node in enumerate(chain):
            kc[b, :, L + d] = k_new[b, node]
            vc[b, :, L + d] = v_new[b, node]
        kl[b] = L + len(chain)
    return kc, vc, kl, status


# ---------------------------------------------------------------------------
# The whole step
# ---------------------------------------------------------------------------

@dataclass
class StepResult:
    u: np.ndarray
    head_logits: np.ndarray
    topk_ids: np.ndarray
    topk_vals: np.ndarray
    topk_margin: np.ndarray
    root: np.ndarray
    tokens: np.ndarray
    positions: np.ndarray
    attn: Optional[np.ndarray]
    logits: np.ndarray
    accept: Dict[str, np.ndarray]
    k_cache: Optional[np.ndarray]
    v_cache: Optional[np.ndarray]
    kv_len: np.ndarray
    commit_status: np.ndarray


def run_step(h, W1, b1, W2, lm_head, X, q, k_new, v_new, k_cache, v_cache, kv_len,
             choices, topk: int, temperature: float, threshold: float = 0.09,
             alpha: float = 0.3, root: Optional[np.ndarray] = None, u_bf16: bool = False,
             attention: bool = True) -> StepResult:
    """One decode step [WIB "Inference flow in an online chat service"]:
    heads and their top-k, tree tokens, tree attention, verification logits,
    typical acceptance and the KV commit of the accepted path.  ``root`` is
    the previous step's next token; None derives it from lm_head(h).
    """
    u, z = medusa_heads(h, W1, b1, W2, u_bf16)
    ids, vals, marg = head_topk(z, topk)
    if root is None:
        root = base_root(h, lm_head)
    tt = tree_tables(choices)
    tok, pos = tree_tokens(tt, np.asarray(root), ids, np.asarray(kv_len))
    D = q.shape[-1]
    attn = (tree_attention(q, k_new, v_new, k_cache, v_cache, kv_len, tt, 1.0 / np.sqrt(D))
            if attention else None)
    logits = verify_logits(X, lm_head)
    acc = typical_accept(logits, tok, tt, temperature, threshold, alpha)
    if k_cache is not None:
        kc, vc, kl, st = kv_commit(k_cache, v_cache, kv_len, k_new, v_new, tt, acc["best_node"])
    else:
        kc = vc = None
        kl, st = np.asarray(kv_len), np.zeros(len(kv_len), np.int64)
    return StepResult(u, z, ids, vals, marg, np.asarray(root), tok, pos, attn, logits, acc,
                      kc, vc, kl, st)
