"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each test states the fact it checks and where it comes from; the expected
values are worked out by hand or come from an independent brute force,
never from the oracle itself.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import read_golden


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------- heads

def test_zero_init_heads_equal_lm_head(golden):
    """Ultralytics "Medusa Heads", PyTorch example: zero FC weights/bias and W2 copied from
    lm_head make every head's logits exactly equal lm_head(h); the page prints [True, True, True]."""
    g = golden("ultralytics_zero_init_heads.txt")
    H, V, K = int(g["hidden_size"][0][0]), int(g["vocab_size"][0][0]), int(g["num_heads"][0][0])
    expected = [s == "True" for s in g["expected"][0]]
    r = _rng(1)
    lm = r.standard_normal((V, H)) * 0.02
    h = r.standard_normal((1, H))
    W1 = np.zeros((K, H, H))
    b1 = np.zeros((K, H))
    W2 = np.broadcast_to(lm, (K, V, H))
    _, z = oracle.medusa_heads(h, W1, b1, W2, u_bf16=False)
    base = oracle.verify_logits(h[:, None, :], lm)[:, 0]
    got = [bool(np.array_equal(z[:, k], base)) for k in range(K)]
    assert got == expected


def test_head_formula_hand_values():
    """u = h + SiLU(W1 h + b1), logits = W2 u (Ultralytics "Medusa Heads": one FC layer with
    SiLU and a residual, then the vocabulary projection).  A non-symmetric W1 catches a
    transposed weight, b1 != 0 a dropped bias, the residual a dropped skip.  Hand values:
    W1 h + b1 = [3 + 0.5, 1 - 1] = [3.5, 0]; SiLU(3.5) = 3.5 / (1 + e^-3.5) = 3.3974071923702527."""
    h = np.array([[1.0, 1.0]])
    W1 = np.array([[[1.0, 2.0], [0.0, 1.0]]])
    b1 = np.array([[0.5, -1.0]])
    W2 = np.array([[[1.0, 0.0], [0.0, 1.0], [1.0, -1.0]]])
    u, z = oracle.medusa_heads(h, W1, b1, W2, u_bf16=False)
    silu35 = 3.3974071923702527
    np.testing.assert_allclose(u[0, 0], [1.0 + silu35, 1.0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(z[0, 0], [1.0 + silu35, 1.0, silu35], rtol=0, atol=1e-14)


def test_silu_negative_branch():
    """SiLU(-1) = -1 / (1 + e) = -0.2689414213699951 (sigmoid gate, not ReLU)."""
    h = np.array([[0.0]])
    u, _ = oracle.medusa_heads(h, np.zeros((1, 1, 1)), np.array([[-1.0]]), np.ones((1, 1, 1)), False)
    assert abs(u[0, 0, 0] - (-0.2689414213699951)) < 1e-15


def test_tree_heads_zero_init_is_the_accepted_rows_verification():
    """Heads over the tree nodes keep the accepted node's row: with the heads' start state
    (W1 = b1 = 0, W2_k = lm_head; Ultralytics "Medusa Heads" example) every head's logits on
    that row equal the verification logits of the accepted node exactly."""
    r = _rng(21)
    B, T, H, V, K = 2, 5, 6, 11, 3
    X = r.standard_normal((B, T, H))
    lm = r.standard_normal((V, H)) * 0.02
    best = np.array([3, 0])
    _, z = oracle.tree_heads(X, best, np.zeros((K, H, H)), np.zeros((K, H)), np.broadcast_to(lm, (K, V, H)), False)
    zv = oracle.verify_logits(X, lm)
    for b in range(B):
        for k in range(K):
            assert np.array_equal(z[b, k], zv[b, best[b]])


def test_tree_heads_reads_only_the_accepted_row():
    """The other tree rows do not enter (changing them leaves the result), and the accepted
    row gives the hand values of the head formula (x = (1, 1) -> u = (1 + SiLU(3.5), 1))."""
    W1 = np.array([[[1.0, 2.0], [0.0, 1.0]]])
    b1 = np.array([[0.5, -1.0]])
    W2 = np.array([[[1.0, 0.0], [0.0, 1.0], [1.0, -1.0]]])
    X = np.array([[[7.0, -3.0], [1.0, 1.0], [0.0, 2.0]]])
    u, z = oracle.tree_heads(X, np.array([1]), W1, b1, W2, False)
    silu35 = 3.3974071923702527
    np.testing.assert_allclose(z[0, 0], [1.0 + silu35, 1.0, silu35], rtol=0, atol=1e-14)
    X2 = X.copy()
    X2[0, [0, 2]] = 99.0
    assert np.array_equal(oracle.tree_heads(X2, np.array([1]), W1, b1, W2, False)[1], z)


def test_bf16_round_known_values():
    """Round-to-nearest-even at bf16's 8 significant bits: 1+2^-8 is a tie -> 1 (even),
    1+3*2^-8 is a tie -> 1+2^-6 (even), 1+2^-8+2^-30 -> 1+2^-7, sign symmetric."""
    x = np.array([1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-30, -(1 + 3 * 2**-8), 3.0, 0.0])
    want = np.array([1.0, 1 + 2**-6, 1 + 2**-7, -(1 + 2**-6), 3.0, 0.0])
    np.testing.assert_array_equal(oracle.bf16_round(x), want)


def test_topk_against_sorted_with_ties():
    """Per-head top-k by brute force: Python's sorted() on (-value, id), ties to the lower id."""
    r = _rng(2)
    z = np.round(r.standard_normal((3, 50)) * 4) / 4     # many exact ties
    ids, vals, _ = oracle.head_topk(z, 7)
    for row in range(3):
        brute = sorted(range(50), key=lambda v: (-z[row, v], v))[:7]
        assert ids[row].tolist() == brute
        assert vals[row].tolist() == [z[row, v] for v in brute]


def test_base_root_is_first_argmax():
    lm = np.array([[1.0], [3.0], [3.0], [2.0]])
    assert oracle.base_root(np.array([[1.0]]), lm).tolist() == [1]


# --------------------------------------------------------------------------- tree

def test_cartesian_2x3_tree(golden):
    """wiblog "Tree attention" worked example: head 1 keeps (It, I), head 2 keeps
    (is, ', the) -> 2 x 3 = 6 candidate paths in a depth-2 tree."""
    g = golden("wiblog_cartesian_2x3.txt")
    head1, head2 = g["head1"][0], g["head2"][0]
    choices = synth.cartesian_choices((len(head1), len(head2)))
    tt = oracle.tree_tables(choices)
    assert len(tt.leaves) == int(g["n_paths"][0][0])
    assert tt.dmax == int(g["depth"][0][0])
    assert tt.T == 1 + 2 + 6
    assert tt.parent.tolist() == [-1, 0, 0, 1, 1, 1, 2, 2, 2]
    vocab = ["<root>"] + head1 + head2
    topk = np.array([[[1, 2, -1], [3, 4, 5]]])          # head1 -> ids 1,2 ; head2 -> ids 3,4,5
    tok, pos = oracle.tree_tokens(tt, np.array([0]), topk, np.array([10]))
    paths = ["|".join(vocab[tok[0, n]] for n in tt.ancestors[leaf][1:] + [leaf]) for leaf in tt.leaves]
    assert paths == g["paths"][0]
    assert pos[0].tolist() == [10, 11, 11, 12, 12, 12, 12, 12, 12]


def test_same_head_tokens_under_every_branch():
    """Ultralytics "Tree attention": head 2 offers the same tokens under every head-1 branch."""
    tt = oracle.tree_tables(synth.cartesian_choices((3, 2)))
    topk = np.array([[[7, 8, 9], [5, 6, 0]]])
    tok, _ = oracle.tree_tokens(tt, np.array([1]), topk, np.array([0]))
    for parent in tt.children[0]:
        assert [tok[0, c] for c in tt.children[parent]] == [5, 6]


def test_single_path_mask_is_causal():
    """wiblog "Tree attention": within one path the mask is the ordinary causal mask."""
    tt = oracle.tree_tables(synth.seeded_sparse_choices(64, (10, 6, 4, 2, 1), 99))
    for leaf in tt.leaves:
        path = tt.ancestors[leaf] + [leaf]
        sub = tt.mask[np.ix_(path, path)]
        assert np.array_equal(sub, np.tril(np.ones((len(path), len(path)), bool)))
    # and different branches never see each other
    a, b = tt.children[0][0], tt.children[0][1]
    assert not tt.mask[a, b] and not tt.mask[b, a]


def test_tree_rejects_bad_choices():
    for bad in ([(0,), (1, 0, 0)], [(0,), (0,)], [()], [(-1,)]):
        with pytest.raises(ValueError):
            oracle.tree_tables(bad)


def test_seeded_tree_invariants():
    """64-node sparse tree, fan-out 10/6/4/2/1: prefix- and rank-closed, depth <= 5."""
    ch = synth.seeded_sparse_choices(64, (10, 6, 4, 2, 1), 1234)
    tt = oracle.tree_tables(ch)
    assert len(ch) == 64 and tt.T == 65 and tt.dmax <= 5
    fan = (10, 6, 4, 2, 1)
    for i in range(tt.T):
        ranks = sorted(tt.rank[c] for c in tt.children[i])
        assert ranks == list(range(len(ranks)))
        assert len(ranks) <= (fan[tt.depth[i]] if tt.depth[i] < 5 else 0)


# --------------------------------------------------------------------------- attention

def _path_attention_brute(q, k_new, v_new, kc, vc, L, path, hq, group, scale):
    """Plain causal attention of one sequence (cache prefix + one path), written out."""
    g = hq // group
    keys = [kc[g, j] for j in range(L)]
    vals = [vc[g, j] for j in range(L)]
    outs = []
    for node in path:
        keys.append(k_new[node, g])
        vals.append(v_new[node, g])
        s = [scale * float(np.dot(q[node, hq], kk)) for kk in keys]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        tot = sum(w)
        outs.append(sum(wi * vv for wi, vv in zip(w, vals)) / tot)
    return outs


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2)])
def test_tree_attention_equals_per_path_causal(Hq, Hkv):
    """Brute force: running every root->leaf path as an ordinary causal sequence after the
    cache must give each node the same output as the tree-masked pass (wiblog "Tree attention")."""
    r = _rng(3)
    choices = synth.cartesian_choices((2, 3))
    tt = oracle.tree_tables(choices)
    B, T, D, L, Lmax = 2, tt.T, 8, 5, 9
    q = r.standard_normal((B, T, Hq, D))
    kn = r.standard_normal((B, T, Hkv, D))
    vn = r.standard_normal((B, T, Hkv, D))
    kc = r.standard_normal((B, Hkv, Lmax, D))
    vc = r.standard_normal((B, Hkv, Lmax, D))
    kv_len = np.array([L, L - 2])
    scale = 1 / math.sqrt(D)
    o = oracle.tree_attention(q, kn, vn, kc, vc, kv_len, tt, scale)
    for b in range(B):
        for leaf in tt.leaves:
            path = tt.ancestors[leaf] + [leaf]
            for hq in range(Hq):
                brute = _path_attention_brute(q[b], kn[b], vn[b], kc[b], vc[b], kv_len[b], path,
                                              hq, Hq // Hkv, scale)
                for node, ob in zip(path, brute):
                    np.testing.assert_allclose(o[b, node, hq], ob, rtol=0, atol=1e-12)


def test_tree_attention_zero_query_is_mean():
    """q = 0 gives equal weights: the output is the mean of the visible values
    (L cache rows plus depth+1 tree rows)."""
    tt = oracle.tree_tables(synth.cartesian_choices((2, 2)))
    r = _rng(4)
    B, T, H, D, L = 1, tt.T, 1, 4, 3
    vn = r.standard_normal((B, T, H, D))
    vc = r.standard_normal((B, H, 6, D))
    o = oracle.tree_attention(np.zeros((B, T, H, D)), r.standard_normal((B, T, H, D)), vn,
                              r.standard_normal((B, H, 6, D)), vc, np.array([L]), tt, 0.5)
    for i in range(T):
        vis = [vc[0, 0, j] for j in range(L)] + [vn[0, a, 0] for a in tt.ancestors[i] + [i]]
        np.testing.assert_allclose(o[0, i, 0], np.mean(vis, axis=0), atol=1e-14)


# --------------------------------------------------------------------------- rotary positions

def test_rope_hand_values():
    """Rotate-half rotary embedding (RoFormer): D = 2, x = (1, 0) at position 1 turns by
    1 radian -> (cos 1, sin 1); D = 4, theta = 10000 at position 2: the pair (x0, x2)
    turns by 2 rad and (x1, x3) by 2 * 10000^(-1/2) = 0.02 rad.  Values written out by hand."""
    got = oracle.apply_rope(np.array([[[1.0, 0.0]]]), np.array([1]), 10000.0)[0, 0]
    np.testing.assert_allclose(got, [0.5403023058681398, 0.8414709848078965], rtol=0, atol=1e-15)
    got = oracle.apply_rope(np.array([[[1.0, 2.0, 3.0, 4.0]]]), np.array([2]), 10000.0)[0, 0]
    want = [-3.1440391170241875, 1.9196053465598233, -0.33914308281574557, 4.039197360052977]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_rope_is_complex_rotation():
    """The same map as multiplying z_d = x_d + i x_(d+D/2) by exp(i p theta^(-2d/D))
    (an independent formulation: a swapped sign or half would fail it)."""
    r = _rng(11)
    x = r.standard_normal((3, 5, 2, 8))
    pos = r.integers(0, 5000, size=(3, 5))
    got = oracle.apply_rope(x, pos, 500.0)
    z = x[..., :4] + 1j * x[..., 4:]
    w = z * np.exp(1j * pos[..., None, None] * 500.0 ** (-(2.0 * np.arange(4)) / 8))
    np.testing.assert_allclose(got, np.concatenate([w.real, w.imag], axis=-1), rtol=0, atol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    """q(m) . k(n) after rotation depends on m - n alone (q and k turned the same way),
    position 0 leaves a vector unchanged, and every rotation keeps the norm."""
    r = _rng(12)
    q, k = r.standard_normal((1, 1, 1, 16)), r.standard_normal((1, 1, 1, 16))
    s = lambda m, n: float(np.sum(oracle.apply_rope(q, np.array([[m]]), 10000.0) *
                                  oracle.apply_rope(k, np.array([[n]]), 10000.0)))
    assert abs(s(7, 3) - s(1007, 1003)) < 1e-10 and abs(s(7, 3) - s(3, 7)) > 1e-3
    np.testing.assert_array_equal(oracle.apply_rope(q, np.array([[0]]), 10000.0), q)
    assert abs(np.linalg.norm(oracle.apply_rope(q, np.array([[123]]), 10000.0)) - np.linalg.norm(q)) < 1e-12


def test_tree_attention_with_positions_equals_rotated_paths():
    """With position ids, every root->leaf path run as a causal sequence after the cache, its
    query and key rows first turned by the complex rotation at positions L + depth, gives each
    node the output of the tree-masked pass."""
    r = _rng(13)
    tt = oracle.tree_tables(synth.cartesian_choices((2, 3)))
    B, T, Hq, Hkv, D, Lmax = 1, tt.T, 2, 1, 8, 9
    q, kn, vn = r.standard_normal((B, T, Hq, D)), r.standard_normal((B, T, Hkv, D)), r.standard_normal((B, T, Hkv, D))
    kc, vc = r.standard_normal((B, Hkv, Lmax, D)), r.standard_normal((B, Hkv, Lmax, D))
    L = 5
    pos = np.array([[L + len(n) for n in tt.nodes]])
    o = oracle.tree_attention(q, kn, vn, kc, vc, np.array([L]), tt, 0.5, positions=pos, rope_theta=100.0)

    def turn(v, p):
        z = v[:4] + 1j * v[4:]
        w = z * np.exp(1j * p * 100.0 ** (-(2.0 * np.arange(4)) / D))
        return np.concatenate([w.real, w.imag])

    qr = np.array([[turn(q[0, i, h], pos[0, i]) for h in range(Hq)] for i in range(T)])[None]
    kr = np.array([[turn(kn[0, i, 0], pos[0, i])] for i in range(T)])[None]
    for leaf in tt.leaves:
        path = tt.ancestors[leaf] + [leaf]
        for hq in range(Hq):
            brute = _path_attention_brute(qr[0], kr[0], vn[0], kc[0], vc[0], L, path, hq, Hq // Hkv, 0.5)
            for node, ob in zip(path, brute):
                np.testing.assert_allclose(o[0, node, hq], ob, rtol=0, atol=1e-12)


def test_verify_logits_hand_values():
    """lm_head [V, H] rows dotted with each tree node's state: rows (1,2),(3,4),(5,6) give
    (1,3,5) for x = (1,0) and (-1,-1,-1) for x = (1,-1)."""
    lm = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])
    X = np.array([[[1.0, 0.0], [1.0, -1.0]]])
    assert oracle.verify_logits(X, lm).tolist() == [[[1.0, 3.0, 5.0], [-1.0, -1.0, -1.0]]]


# --------------------------------------------------------------------------- acceptance

def test_uniform_logits_closed_form(golden):
    """Uniform logits: p = 1/V and H = ln V, so the effective threshold is
    min(0.09, 0.3/V) and the candidate is accepted (typical acceptance, wiblog; defaults cnnetsun)."""
    g = golden("cnnetsun_posterior_defaults.txt")
    thr, alpha = float(g["posterior_threshold"][0][0]), float(g["posterior_alpha"][0][0])
    assert abs(alpha - math.sqrt(thr)) < 1e-15
    for V in (2, 3, 1000, 32000):
        r = oracle.node_posterior(np.full(V, 1.7), 1, 0.7, thr, alpha)
        assert abs(r["p"] - 1 / V) < 1e-15
        assert abs(r["H"] - math.log(V)) < 1e-12
        assert abs(r["thr"] - min(0.09, 0.3 / V)) < 1e-15
        assert r["accept"]


def test_posterior_hand_example():
    """q = (0.1, 0.2, 0.7): H = 0.8018185525433373, alpha*exp(-H) = 0.13455... so with
    threshold 0.09 every token passes, with threshold 0.15 the 0.1 token fails.
    (The effective threshold is the MIN of the hard and the entropy threshold, wiblog.)"""
    z = np.log(np.array([0.1, 0.2, 0.7]))
    H = -(0.1 * math.log(0.1) + 0.2 * math.log(0.2) + 0.7 * math.log(0.7))
    assert abs(H - 0.8018185525433373) < 1e-15
    for t, exp_p in enumerate((0.1, 0.2, 0.7)):
        r = oracle.node_posterior(z, t, 1.0, 0.09, 0.3)
        assert abs(r["p"] - exp_p) < 1e-14 and abs(r["H"] - H) < 1e-14 and r["accept"]
    r0 = oracle.node_posterior(z, 0, 1.0, 0.15, 0.3)
    assert abs(r0["thr"] - 0.3 * math.exp(-H)) < 1e-15 and not r0["accept"]
    assert oracle.node_posterior(z, 1, 1.0, 0.15, 0.3)["accept"]


def test_one_hot_dominant():
    z = np.zeros(100)
    z[42] = 50.0
    assert oracle.node_posterior(z, 42, 0.7, 0.09, 0.3)["accept"]
    assert not oracle.node_posterior(z, 41, 0.7, 0.09, 0.3)["accept"]


def test_temperature_zero_is_greedy_and_limit():
    """wiblog "Typical acceptance": at temperature zero it reduces to greedy decoding.
    Also the limit: a tiny temperature with a clear top-1 margin decides the same way."""
    r = _rng(5)
    for _ in range(20):
        z = r.standard_normal(64) * 3
        s = np.sort(z)
        if s[-1] - s[-2] < 0.05:
            continue
        top = int(np.argmax(z))
        for t in range(64):
            g0 = oracle.node_posterior(z, t, 0.0, 0.09, 0.3)["accept"]
            assert g0 == (t == top)
            assert oracle.node_posterior(z, t, 1e-3, 0.09, 0.3)["accept"] == g0
    zt = np.array([1.0, 5.0, 5.0, 0.0])                  # greedy tie -> lowest id
    assert oracle.node_posterior(zt, 1, 0.0, 0.09, 0.3)["accept"]
    assert not oracle.node_posterior(zt, 2, 0.0, 0.09, 0.3)["accept"]


def test_threshold_falls_as_temperature_rises():
    """wiblog "How the acceptance rate shapes the speedup": a higher temperature raises the
    entropy, so the entropy threshold (and thus min(thr, alpha e^-H)) falls."""
    r = _rng(6)
    z = r.standard_normal(500) * 2
    thr = [oracle.node_posterior(z, 0, t, 0.09, 0.3)["thr"] for t in (0.2, 0.5, 0.7, 1.0, 2.0)]
    assert all(a >= b for a, b in zip(thr, thr[1:]))
    assert thr[-1] < thr[0]


def _tree_logits(tt, tokens, V, accept_children):
    """Logits where exactly the listed children are the parent's greedy choice."""
    z = np.zeros((1, tt.T, V))
    for c in accept_children:
        z[0, tt.parent[c], tokens[0, c]] = 10.0
    return z


def test_longest_prefix_and_tie_break():
    """Longest accepted branch wins (ULT); a node counts only if its parent is kept; among
    equally deep kept nodes the first in canonical order wins; the root is always kept (wiblog)."""
    tt = oracle.tree_tables(synth.cartesian_choices((2, 3)))
    # nodes: 0 root; 1 (0,) 2 (1,); 3 (0,0) 4 (0,1) 5 (0,2) 6 (1,0) 7 (1,1) 8 (1,2)
    tokens = np.array([[0, 11, 12, 21, 22, 23, 21, 22, 23]])
    V = 30
    # (a) temperature 0.7: the root splits its mass between tokens 11 and 12, so both depth-1
    #     nodes pass; children 4 (under 1) and 7 (under 2) pass too -> equal depth, node 4 first
    z = _tree_logits(tt, tokens, V, [1, 4, 7])
    z[0, 0, 12] = 10.0
    acc = oracle.typical_accept(z, tokens, tt, 0.7, 0.09, 0.3)
    assert acc["node_accept"][0].tolist() == [True, True, True, False, True, False, False, True, False]
    assert acc["best_node"][0] == 4 and acc["accept_len"][0] == 2
    assert acc["accepted_tokens"][0].tolist() == [0, 11, 22]
    assert acc["best_path"][0] == 1                      # leaves are 3..8 -> path index 1 is node 4
    # (a') temperature 0 with the same greedy tie: the lowest id (11) is the greedy token, so
    #      node 2 fails and its child 7 cannot count
    acc = oracle.typical_accept(z, tokens, tt, 0.0, 0.09, 0.3)
    assert acc["node_accept"][0].tolist() == [True, True, False, False, True, False, False, False, False]
    # (b) a deep child whose parent fails does not count
    z = _tree_logits(tt, tokens, V, [5])
    z[0, 0, 29] = 10.0
    acc = oracle.typical_accept(z, tokens, tt, 0.0, 0.09, 0.3)
    assert acc["accept_len"][0] == 0 and acc["best_node"][0] == 0
    assert acc["accepted_tokens"][0].tolist() == [0, -1, -1]
    assert acc["next_root"][0] == 29                     # greedy token of the winner (the root)
    assert acc["best_path"][0] == 0                      # every path runs through the root
    # (b') an inner winner: node 2 passes, none of its children does -> the first path through
    #      it is the one ending at its first child, node 6 (path index 3)
    z = _tree_logits(tt, tokens, V, [2])
    z[0, 2, 29] = 10.0
    acc = oracle.typical_accept(z, tokens, tt, 0.0, 0.09, 0.3)
    assert acc["best_node"][0] == 2 and acc["accept_len"][0] == 1 and acc["best_path"][0] == 3
    assert acc["accepted_tokens"][0].tolist() == [0, 12, -1] and acc["next_root"][0] == 29
    # (c) temperature > 0 with one clear branch
    z = _tree_logits(tt, tokens, V, [2, 8])
    acc = oracle.typical_accept(z * 3, tokens, tt, 0.7, 0.09, 0.3)
    assert acc["best_node"][0] == 8 and acc["accept_len"][0] == 2


# --------------------------------------------------------------------------- commit

def test_joint_probability_tie_break_hand_example():
    """Among equally deep kept nodes, the tie-break by highest joint probability (the
    product of each node's p under its parent) against first-in-canonical-order, on a
    hand-built 2 x 3 tree at temperature 1.  Tokens: root 0, depth 1 (0,)->1, (1,)->2,
    depth 2 ranks 0,1,2 -> tokens 3,4,5 under both.  exp(logits): root [1,3,1,1,1,1]
    (p(1) = 3/8, p(2) = 1/8, H = 1.6675, threshold 0.0566: both kept); node (0,)
    [1,1,1,2,1,1] (2/7, 1/7, 1/7 against 0.0522: all kept); node (1,) [1,1,1,1,1,40]
    (1/45, 1/45, 40/45 against min(0.09, 0.177) = 0.09: only (1,2) kept).  Joint
    probabilities of the depth-2 survivors: (0,0) 3/8 * 2/7 = 0.1071, (0,1) = (0,2) =
    0.0536, (1,2) 1/8 * 40/45 = 0.1111.  First-in-order picks (0,0), node 3; joint picks
    (1,2), node 8."""
    tt = oracle.tree_tables(synth.cartesian_choices((2, 3)))
    assert tt.nodes[3] == (0, 0) and tt.nodes[8] == (1, 2)
    tokens = np.array([[0, 1, 2, 3, 4, 5, 3, 4, 5]])
    z = np.zeros((1, tt.T, 6))
    z[0, 0] = np.log([1, 3, 1, 1, 1, 1])
    z[0, 1] = np.log([1, 1, 1, 2, 1, 1])
    z[0, 2] = np.log([1, 1, 1, 1, 1, 40])
    first = oracle.typical_accept(z, tokens, tt, 1.0, 0.09, 0.3)
    joint = oracle.typical_accept(z, tokens, tt, 1.0, 0.09, 0.3, tie_break="joint")
    assert first["accept_len"][0] == joint["accept_len"][0] == 2
    assert first["best_node"][0] == 3 and joint["best_node"][0] == 8
    assert joint["accepted_tokens"][0].tolist() == [0, 2, 5]
    assert abs(joint["joint_margin"][0] - (math.log(40 / 360) - math.log(6 / 56))) < 1e-12
    # at temperature 0 every kept node has p = 1: the joint rule falls back to the order
    g0 = oracle.typical_accept(z, tokens, tt, 0.0, 0.09, 0.3, tie_break="joint")
    f0 = oracle.typical_accept(z, tokens, tt, 0.0, 0.09, 0.3)
    assert g0["best_node"][0] == f0["best_node"][0]


def test_nucleus_hand_example():
    """q = (0.1, 0.2, 0.7) (logits ln q, temperature 1), top_p = 0.75: by descending
    probability 0.7 < 0.75, then 0.7 + 0.2 = 0.9 >= 0.75, so the nucleus is tokens {1, 2}
    with mass 0.9.  In id order the running mass is 0.2, 0.9: u = 0.2 -> target 0.18 ->
    token 1; u = 0.5 -> target 0.45 -> token 2; u = 0.99 -> token 2."""
    z = np.log([0.1, 0.2, 0.7])
    for u, want in ((0.2, 1), (0.5, 2), (0.99, 2)):
        r = oracle.nucleus_next(z, 1.0, 0.75, u)
        assert (r["token"], r["size"]) == (want, 2)
    assert oracle.nucleus_next(z, 1.0, 0.75, 0.2)["margin"] > 0.01


def test_nucleus_limits():
    """top_p -> 0+ keeps only the most probable token (greedy for every draw); top_p = 1
    keeps every token, and the draw then follows the plain inverse CDF (brute force over a
    cumulative sum in id order); temperature 0 is the greedy token."""
    r = _rng(31)
    z = r.standard_normal(50) * 2
    top = int(np.argmax(z))
    for u in (0.0, 0.3, 0.999):
        assert oracle.nucleus_next(z, 0.7, 1e-9, u)["token"] == top
    q = np.exp(z / 0.7 - np.max(z / 0.7))
    q /= q.sum()
    for u in (0.01, 0.37, 0.8):
        brute = next(i for i, c in enumerate(np.cumsum(q)) if c > u)
        assert oracle.nucleus_next(z, 0.7, 1.0, u)["token"] == brute
    assert oracle.nucleus_next(z, 0.0, 0.9, 0.5)["token"] == top


def test_kv_commit_rows_and_overflow():
    tt = oracle.tree_tables(synth.cartesian_choices((2, 3)))
    r = _rng(7)
    B, Hkv, Lmax, D = 2, 2, 12, 4
    kc = r.standard_normal((B, Hkv, Lmax, D))
    vc = r.standard_normal((B, Hkv, Lmax, D))
    kn = r.standard_normal((B, tt.T, Hkv, D))
    vn = r.standard_normal((B, tt.T, Hkv, D))
    kv_len = np.array([5, 10])
    best = np.array([7, 4])                              # path root -> 2 -> 7 ; root -> 1 -> 4
    k2, v2, kl, st = oracle.kv_commit(kc, vc, kv_len, kn, vn, tt, best)
    assert kl.tolist() == [8, 10] and st.tolist() == [0, 1]
    for d, node in enumerate([0, 2, 7]):
        assert np.array_equal(k2[0, :, 5 + d], kn[0, node]) and np.array_equal(v2[0, :, 5 + d], vn[0, node])
    untouched = [j for j in range(Lmax) if not 5 <= j < 8]
    assert np.array_equal(k2[0, :, untouched], kc[0, :, untouched])
    assert np.array_equal(k2[1], kc[1]) and np.array_equal(v2[1], vc[1])


# --------------------------------------------------------------------------- whole step

def test_tiny_step_runs_and_is_consistent():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, variant="plant", plant_depth=2)
    n = lambda t: t.to(torch.float64).numpy()
    res = oracle.run_step(n(inp.h), n(inp.W1), n(inp.b1), n(inp.W2), n(inp.lm_head), n(inp.X),
                          n(inp.q), n(inp.k_new), n(inp.v_new), n(inp.k_cache), n(inp.v_cache),
                          inp.kv_len.numpy(), inp.choices, wl.k_needed(), 0.7,
                          root=inp.root.numpy())
    # the planted tokens are the heads' top-1 and the planted chain is accepted
    assert res.topk_ids[0, 0, 0] == inp.plant["tokens"][0][0]
    assert res.accept["accept_len"][0] >= 2
    assert res.kv_len[0] == wl.L + res.accept["accept_len"][0] + 1


# --------------------------------------------------------------------------- synth

def test_splitmix64_reference_vectors(golden):
    g = golden("splitmix64_vectors.txt")
    for row in g["seed"]:
        seed = int(row[0])
        want = [int(x) for x in row[2:]]
        assert [synth.splitmix64_py(seed, i) for i in range(len(want))] == want


def test_counter_generator_matches_python_mix():
    """The vectorised int64 splitmix64 equals the Python-integer one, element by element."""
    seed = synth.tensor_seed(3, 9)
    idx = torch.tensor([0, 1, 2, 12345, 2**33 + 7])
    x = synth.normal_at(seed, idx, 1.0)
    for e, val in zip(idx.tolist(), x.tolist()):
        s = 0
        for j in range(3):
            z = synth.splitmix64_py(seed, 3 * e + j)
            s += sum((z >> sh) & 0xFFFF for sh in (0, 16, 32, 48))
        assert val == (s - 393210) / 65536.0
