"""Whole-step checks against the oracle on workloads too large for the oracle to
compute every output: every head logit and commit row exactly, attention
outputs and verification logits on seeded samples, and the acceptance cascade
along the nodes it actually reaches.  Shared by the full-size parity tests and
the tests of the timed (logits-free) configuration."""
import math

import numpy as np
import torch

import oracle
from _util import DELTA, TOL, check_topk, np64, npi, rel_err


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check_heads(wl, inp, step):
    kind = wl.dtype
    h = _f64(inp.h)
    near = 0
    k = wl.k_needed()
    for head in range(wl.K):
        _, z = oracle.medusa_heads(h, _f64(inp.W1[head:head + 1]), _f64(inp.b1[head:head + 1]),
                                   _f64(inp.W2[head:head + 1]), u_bf16=(kind == "bf16"))
        if step.head_logits is not None:
            assert rel_err(step.head_logits[:, head], z[:, 0]) < TOL[kind], head
        near += check_topk(step.topk_ids[:, head], step.topk_vals[:, head], z[:, 0], k, DELTA[kind])
    return near


def check_tree(wl, inp, step, tt):
    tok, pos = oracle.tree_tokens(tt, npi(step.root), npi(step.topk_ids), npi(inp.kv_len))
    assert np.array_equal(npi(step.tokens), tok)
    assert np.array_equal(npi(step.positions), pos)


def check_attention(wl, inp, step, tt, n=192, seed=5):
    rng = np.random.default_rng(seed)
    picks = {(int(rng.integers(wl.B)), int(rng.integers(tt.T)), int(rng.integers(wl.Hq))) for _ in range(n)}
    deepest = int(np.argmax(tt.depth))
    picks |= {(b, deepest, wl.Hq - 1) for b in range(wl.B)} | {(b, 0, 0) for b in range(wl.B)}
    picks = sorted(picks)
    o = {}
    for b in sorted({p[0] for p in picks}):
        sel = [(0, i, hq) for (bb, i, hq) in picks if bb == b]
        L = int(inp.kv_len[b])
        a = oracle.tree_attention(_f64(inp.q[b:b + 1]), _f64(inp.k_new[b:b + 1]), _f64(inp.v_new[b:b + 1]),
                                  _f64(inp.k_cache[b:b + 1, :, :L]), _f64(inp.v_cache[b:b + 1, :, :L]),
                                  np.array([L]), tt, 1.0 / math.sqrt(wl.D), only=sel)
        for (_, i, hq) in sel:
            o[(b, i, hq)] = a[0, i, hq]
    got = np.stack([np64(step.attn_out[b, i, hq]) for (b, i, hq) in picks])
    want = np.stack([o[p] for p in picks])
    assert rel_err(got, want) < TOL[wl.dtype]


class LazyLogits:
    """Verification logit rows computed on demand in fp64 (lm_head converted in row chunks)."""

    def __init__(self, X, lm_head):
        self.X = X
        self.lm = lm_head
        self.rows = {}

    def fill(self, keys):
        keys = [k for k in dict.fromkeys(keys) if k not in self.rows]
        if not keys:
            return
        xs = np.stack([_f64(self.X[b, i]) for (b, i) in keys])
        V = self.lm.shape[0]
        z = np.empty((len(keys), V))
        for v0 in range(0, V, 16384):
            z[:, v0:v0 + 16384] = oracle.verify_logits(xs[:, None, :], _f64(self.lm[v0:v0 + 16384]))[:, 0]
        for k, row in zip(keys, z):
            self.rows[k] = row


def check_verify_accept(wl, inp, step, tt, temperature, sample_rows=4, seed=9):
    """Logit rows of sampled nodes, then the acceptance cascade along the nodes it reaches."""
    kind, delta = wl.dtype, DELTA[wl.dtype]
    lz = LazyLogits(inp.X, inp.lm_head)
    rng = np.random.default_rng(seed)
    sampled = [(int(rng.integers(wl.B)), int(rng.integers(tt.T))) for _ in range(sample_rows)]
    lz.fill(sampled)
    if step.logits is not None:
        for (b, i) in sampled:
            assert rel_err(step.logits[b, i], lz.rows[(b, i)]) < TOL[kind]
    tokens = npi(step.tokens)
    near = 0
    for b in range(wl.B):
        # evaluate the cascade top-down, computing the rows of every node it can reach
        frontier = [0]
        while frontier:
            lz.fill([(b, n) for n in frontier])
            nxt = []
            for n in frontier:
                for c in tt.children[n]:
                    r = oracle.node_posterior(lz.rows[(b, n)], int(tokens[b, c]), temperature,
                                              wl.posterior_threshold, wl.posterior_alpha)
                    tie = r["margin"] < (delta / temperature if temperature > 0 else
                                         delta * max(1.0, abs(lz.rows[(b, n)]).max()))
                    if (r["accept"] or tie) and tt.children[c]:
                        nxt.append(c)
                    elif r["accept"] or tie:
                        lz.fill([(b, c)])
            frontier = nxt
        best_g = int(step.best_node[b])
        lz.fill([(b, best_g)])
        z = np.full((1, tt.T, wl.V), np.nan)
        for (bb, i), row in lz.rows.items():
            if bb == b:
                z[0, i] = row
        with np.errstate(invalid="ignore"):
            acc = oracle.typical_accept(z, tokens[b:b + 1], tt, temperature, wl.posterior_threshold,
                                        wl.posterior_alpha)
        m = acc["margin"][0][1:]
        m = np.where(np.isnan(m), np.inf, m)
        tie = m.min() < (delta / temperature if temperature > 0 else delta * 10) if m.size else False
        same = (int(step.accept_len[b]) == acc["accept_len"][0] and best_g == acc["best_node"][0]
                and int(step.best_path[b]) == acc["best_path"][0]
                and npi(step.accepted_tokens[b]).tolist() == acc["accepted_tokens"][0].tolist())
        if not same:
            assert tie, (b, int(step.accept_len[b]), acc["accept_len"][0])
            near += 1
        else:
            srt = np.sort(z[0, best_g])
            if int(step.next_root[b]) != acc["next_root"][0]:
                assert srt[-1] - srt[-2] < delta * max(1.0, abs(srt[-1]))
                near += 1
    return near


def check_commit(wl, inp, step, kc, vc, kl, tt):
    kv0 = npi(inp.kv_len)
    for b in range(wl.B):
        best = int(step.best_node[b])
        chain = tt.ancestors[best] + [best]
        L = int(kv0[b])
        if L + len(chain) > wl.Lmax:
            assert int(kl[b]) == L
            continue
        assert int(kl[b]) == L + len(chain)
        for d, node in enumerate(chain):
            assert torch.equal(kc[b, :, L + d], inp.k_new[b, node])
            assert torch.equal(vc[b, :, L + d], inp.v_new[b, node])
        assert torch.equal(kc[b, :, :L], inp.k_cache[b, :, :L])
        assert torch.equal(kc[b, :, L + len(chain):], inp.k_cache[b, :, L + len(chain):])


