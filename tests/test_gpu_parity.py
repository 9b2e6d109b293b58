"""GPU parity: the CUDA path through the C ABI against the CPU oracle,
element by element, on the same seeded inputs (small and 7B-shaped workloads).

Stage by stage: each stage's oracle runs on the GPU's (already checked)
discrete outputs of the stage before, so a near-tie upstream (counted, not
failed) never masks a real mismatch downstream.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import (DELTA, SMALL_BF16, SMALL_BF16_D64, SMALL_BF16_G3, TOL, accept_parity, check_topk, np64, npi,
                   rel_err, step_oracle_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mb():
    assert torch.cuda.is_available(), "the CUDA parity tests need a GPU"
    import medusa_head_speculative_04_b300 as m
    return m


def make_step(mb, wl, inp, root_from_lm=False, **kw):
    return mb.MedusaStep(inp.choices, wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.k_needed(),
                         inp.dtype, root_from_lm_head=root_from_lm, keep_head_logits=True, keep_logits=True,
                         **kw)


def run_step(mb, wl, inp, temperature, root_from_lm=False, **kw):
    step = make_step(mb, wl, inp, root_from_lm, **kw)
    kc, vc, kl = inp.k_cache.clone(), inp.v_cache.clone(), inp.kv_len.clone()
    step.run(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, inp.X, inp.q, inp.k_new, inp.v_new, kc, vc, kl,
             temperature, wl.posterior_threshold, wl.posterior_alpha, root=inp.root)
    torch.cuda.synchronize()
    return step, kc, vc, kl


def check_full(wl, inp, step, kc, vc, kl, temperature, root_from_lm=False, tie_break="first"):
    """Whole-step parity with the oracle computing every output."""
    kind = wl.dtype
    tol, delta = TOL[kind], DELTA[kind]
    o = step_oracle_inputs(inp)
    near = 0
    # heads + top-k
    _, z_o = oracle.medusa_heads(o["h"], o["W1"], o["b1"], o["W2"], u_bf16=(kind == "bf16"))
    assert rel_err(step.head_logits, z_o) < tol
    k = wl.k_needed()
    near += check_topk(step.topk_ids, step.topk_vals, z_o, k, delta)
    ids = npi(step.topk_ids)
    vals_o = np.take_along_axis(z_o, ids, axis=-1)
    assert rel_err(step.topk_vals, vals_o) < tol
    if root_from_lm:
        z_root = o["h"] @ o["lm_head"].T
        for b in range(wl.B):
            g, r = int(step.root[b]), int(oracle.base_root(o["h"][b:b + 1], o["lm_head"])[0])
            if g != r:
                assert abs(z_root[b, g] - z_root[b, r]) < delta * max(1.0, abs(z_root[b, r]))
                near += 1
    # tree
    tt = oracle.tree_tables(inp.choices)
    root = npi(step.root)
    tok_o, pos_o = oracle.tree_tokens(tt, root, ids, npi(inp.kv_len))
    assert np.array_equal(npi(step.tokens), tok_o)
    assert np.array_equal(npi(step.positions), pos_o)
    cand = npi(step.candidates)
    for p, leaf in enumerate(tt.leaves):
        chain = tt.ancestors[leaf] + [leaf]
        want = np.full(tt.dmax + 1, -1)
        for b in range(wl.B):
            want[: len(chain)] = tok_o[b, chain]
            assert cand[b, p].tolist() == want.tolist()
    # attention
    a_o = oracle.tree_attention(o["q"], o["k_new"], o["v_new"], o["k_cache"], o["v_cache"], npi(inp.kv_len), tt,
                                1.0 / math.sqrt(wl.D))
    assert rel_err(step.attn_out, a_o) < tol
    # verification logits + acceptance
    zv = oracle.verify_logits(o["X"], o["lm_head"])
    assert rel_err(step.logits, zv) < tol
    near += accept_parity(step, zv, npi(step.tokens), tt, temperature, wl.posterior_threshold,
                          wl.posterior_alpha, delta, kind, tie_break=tie_break)
    if temperature > 0:
        H_o = np.array([[oracle.node_posterior(zv[b, i], 0, temperature, 0.09, 0.3)["H"] for i in range(tt.T)]
                        for b in range(wl.B)])
        assert rel_err(step.node_H, H_o) < max(tol, 1e-3)
    # commit (bit-exact on the GPU's own decision)
    kc_o, vc_o, kl_o, st_o = oracle.kv_commit(o["k_cache"], o["v_cache"], npi(inp.kv_len), o["k_new"],
                                              o["v_new"], tt, npi(step.best_node))
    assert np.array_equal(npi(kl), kl_o)
    assert np.array_equal(np64(kc), kc_o) and np.array_equal(np64(vc), vc_o)
    st = npi(step.dev_status)
    assert np.array_equal(st & 1, st_o), st
    assert np.all((st & ~1) == 0), st
    return near


# ----------------------------------------------------------------------------- generator


def test_generator_bit_identical_on_gpu():
    seed = synth.tensor_seed(7, 3)
    for dt in (torch.float32, torch.bfloat16):
        a = synth.normal((3, 1000, 37), seed, 0.02, dt, "cpu")
        b = synth.normal((3, 1000, 37), seed, 0.02, dt, "cuda").cpu()
        assert torch.equal(a.view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                           b.view(torch.int16 if dt == torch.bfloat16 else torch.int32))


# ----------------------------------------------------------------------------- tiny (fp32)

@pytest.mark.parametrize("variant", ["random", "plant", "zeroinit"])
@pytest.mark.parametrize("temperature", [0.0, 0.7])
def test_tiny_full_step(mb, variant, temperature, near_ties):
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, "cuda", variant=variant, plant_depth=2)
    step, kc, vc, kl = run_step(mb, wl, inp, temperature)
    near = near_ties(check_full(wl, inp, step, kc, vc, kl, temperature))
    assert near <= 2
    if variant == "plant":
        assert int(step.accept_len[0]) == 2


@pytest.mark.parametrize("name", ["tiny", "vicuna7b"])
def test_root_from_lm_head(mb, name, near_ties):
    """The root as argmax lm_head(h), an extra block of the vocabulary launch: at the 7B
    shape that launch hands its rows out dynamically, at the tiny one it splits them
    statically."""
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda")
    step, kc, vc, kl = run_step(mb, wl, inp, 0.7, root_from_lm=True)
    assert near_ties(check_full(wl, inp, step, kc, vc, kl, 0.7, root_from_lm=True)) <= 2


@pytest.mark.parametrize("name", ["tiny", "vicuna7b"])
def test_zero_init_heads_bitwise(mb, name):
    """Ultralytics "Medusa Heads" example: with zero FC weights and W2 = lm_head every head
    reproduces lm_head(h) exactly -- on the GPU: every head's logits are bitwise identical, and
    each head's top-1 is the root the lm_head path picks."""
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda", variant="zeroinit")
    step = make_step(mb, wl, inp, root_from_lm=True)
    step.heads(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head)
    torch.cuda.synchronize()
    hl = step.head_logits
    for k in range(1, wl.K):
        assert torch.equal(hl[:, k], hl[:, 0])
    assert torch.equal(step.topk_ids[:, :, 0], step.root[:, None].expand(-1, wl.K))
    o = step_oracle_inputs(inp)
    z_base = o["h"] @ o["lm_head"].T
    assert rel_err(hl[:, 0], z_base) < TOL[wl.dtype]


# ----------------------------------------------------------------------------- small bf16, multi-tile



def test_zero_init_heads_bitwise_tensor_core_path(mb):
    """The same example at three batch rows with the root given, where z_k = W2_k u_k runs
    as one grouped tcgen05 GEMM: every head's logits are still bitwise identical."""
    wl = SMALL_BF16
    inp = synth.make_inputs(wl, "cuda", variant="zeroinit")
    step = make_step(mb, wl, inp)
    step.heads(inp.h, inp.W1, inp.b1, inp.W2)
    torch.cuda.synchronize()
    hl = step.head_logits
    for k in range(1, wl.K):
        assert torch.equal(hl[:, k], hl[:, 0])
        assert torch.equal(step.topk_ids[:, k], step.topk_ids[:, 0])
    o = step_oracle_inputs(inp)
    assert rel_err(hl[:, 0], o["h"] @ o["lm_head"].T) < TOL[wl.dtype]


@pytest.mark.parametrize("wl", [SMALL_BF16, SMALL_BF16_D64, SMALL_BF16_G3], ids=lambda w: w.name)
@pytest.mark.parametrize("temperature", [0.0, 0.7])
@pytest.mark.parametrize("variant", ["random", "plant"])
def test_small_bf16_full_step(mb, wl, temperature, variant, near_ties):
    """Ragged kv lengths (including 0), a vocabulary that is not a multiple of any tile,
    GQA (groups 4 and 3: both attention kernels), several requests, both head dims."""
    inp = synth.make_inputs(wl, "cuda", variant=variant)
    step, kc, vc, kl = run_step(mb, wl, inp, temperature)
    near = near_ties(check_full(wl, inp, step, kc, vc, kl, temperature))
    assert near <= 3


def test_captured_step_replays_new_inputs(mb, near_ties):
    """MedusaStep.capture: a graph replay after the captured tensors are refilled in place
    computes the step of the new contents (checked against the oracle)."""
    wl = SMALL_BF16
    inp = synth.make_inputs(wl, "cuda", variant="plant")
    step = make_step(mb, wl, inp)
    kc, vc, kl0 = inp.k_cache.clone(), inp.v_cache.clone(), inp.kv_len.clone()
    kl = kl0.clone()
    act = {k: getattr(inp, k).clone() for k in ("h", "X", "q", "k_new", "v_new", "root")}
    g = step.capture(act["h"], inp.W1, inp.b1, inp.W2, inp.lm_head, act["X"], act["q"], act["k_new"],
                     act["v_new"], kc, vc, kl, 0.7, wl.posterior_threshold, wl.posterior_alpha, root=act["root"],
                     prologue=lambda: kl.copy_(kl0))
    other = synth.make_inputs(dataclasses.replace(wl, config_id=14), "cuda", variant="random")
    for k in act:
        act[k].copy_(getattr(other, k))
    kc.copy_(inp.k_cache)
    vc.copy_(inp.v_cache)
    for t in (step.results, step.attn_out, step.logits, step.head_logits, step.dev_status):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    mixed = dataclasses.replace(inp, **{k: getattr(other, k) for k in act}, plant=None)
    near = near_ties(check_full(wl, mixed, step, kc, vc, kl, 0.7))
    assert near <= 3


def test_root_only_tree(mb):
    """Degenerate tree without candidates: only the root is emitted, accept_length 0."""
    wl = dataclasses.replace(synth.WORKLOADS["tiny"], name="root_only", tree=("cartesian", ()))
    inp = synth.make_inputs(wl, "cuda")
    assert inp.choices == [] and inp.T == 1
    step, kc, vc, kl = run_step(mb, wl, inp, 0.7)
    assert int(step.accept_len[0]) == 0 and int(step.best_node[0]) == 0
    assert int(kl[0]) == wl.L + 1
    check_full(wl, inp, step, kc, vc, kl, 0.7)


def test_kv_overflow_flag_leaves_cache(mb):
    wl = dataclasses.replace(synth.WORKLOADS["tiny"], name="overflow", lmax_slack=1)
    inp = synth.make_inputs(wl, "cuda", variant="plant", plant_depth=2)
    step, kc, vc, kl = run_step(mb, wl, inp, 0.7)
    assert int(step.accept_len[0]) == 2
    assert int(step.dev_status[0]) & mb.DEV_KV_OVERFLOW
    assert int(kl[0]) == wl.L
    assert torch.equal(kc, inp.k_cache) and torch.equal(vc, inp.v_cache)


# ----------------------------------------------------------------------------- 7B shape, full size

@pytest.mark.parametrize("temperature", [0.0, 0.7])
@pytest.mark.parametrize("variant", ["plant", "random"])
def test_vicuna7b_full_step(mb, temperature, variant, near_ties):
    wl = synth.WORKLOADS["vicuna7b"]
    inp = synth.make_inputs(wl, "cuda", variant=variant)
    step, kc, vc, kl = run_step(mb, wl, inp, temperature, kv_len_hint=wl.L)
    near = near_ties(check_full(wl, inp, step, kc, vc, kl, temperature))
    assert near <= 3
    if variant == "plant":
        assert int(step.accept_len[0]) >= inp.plant["depths"][0]


# ----------------------------------------------------------------------------- device status

def test_nan_hidden_state_flags_its_request_only(mb):
    """A NaN in one tree node's hidden state (request 1, a leaf off the planted path) makes
    that node's logits NaN: the request is flagged MEDUSA_DEV_NAN, the other requests are
    not, and every acceptance output equals the clean step's (the leaf has no children and
    does not win)."""
    wl = SMALL_BF16
    inp = synth.make_inputs(wl, "cuda", variant="plant")
    clean, _, _, _ = run_step(mb, wl, inp, 0.7)
    tt = oracle.tree_tables(inp.choices)
    leaf = tt.nodes.index((2, 1, 1))
    assert not tt.children[leaf] and int(clean.best_node[1]) != leaf
    X = inp.X.clone()
    X[1, leaf, 7] = float("nan")
    bad = dataclasses.replace(inp, X=X)
    step, kc, vc, kl = run_step(mb, wl, bad, 0.7)
    st = npi(step.dev_status)
    assert st[1] & mb.DEV_NAN and st[0] == 0 and st[2] == 0, st
    assert torch.equal(step.results, clean.results)
    assert torch.isnan(step.logits[1, leaf]).all()
    other = [i for i in range(tt.T) if i != leaf]
    assert torch.equal(step.logits[:, other], clean.logits[:, other])


def test_missing_candidate_flags_bad_token(mb):
    """A top-k entry of -1 (no candidate) reaching the tree expansion sets
    MEDUSA_DEV_BAD_TOKEN for that request only; the other request's tokens are exact."""
    wl = dataclasses.replace(SMALL_BF16, B=2)
    inp = synth.make_inputs(wl, "cuda")
    tt = oracle.tree_tables(inp.choices)
    k = wl.k_needed()
    ids = torch.arange(wl.B * wl.K * k, dtype=torch.int32, device="cuda").view(wl.B, wl.K, k).contiguous()
    ids[0, 1, 1] = -1                     # head 2, rank 1 of request 0: used by nodes (r, 1)
    T, P, W = tt.T, len(tt.leaves), tt.dmax + 1
    tokens = torch.zeros(wl.B, T, dtype=torch.int32, device="cuda")
    pos = torch.zeros_like(tokens)
    cand = torch.zeros(wl.B, P, W, dtype=torch.int32, device="cuda")
    st = torch.zeros(wl.B, dtype=torch.int32, device="cuda")
    tree = mb.Tree(inp.choices)
    mb.medusa_build_tree(tree, inp.root, ids, inp.kv_len, tokens, pos, cand, st)
    torch.cuda.synchronize()
    assert int(st[0]) == mb.DEV_BAD_TOKEN and int(st[1]) == 0
    tok_o, pos_o = oracle.tree_tokens(tt, npi(inp.root), npi(ids), npi(inp.kv_len))
    assert np.array_equal(npi(tokens), tok_o)       # the -1 is passed through, not replaced
    assert np.array_equal(npi(pos), pos_o)


# ----------------------------------------------------------------------------- positions

def test_tree_query_sizes(mb):
    """medusa_tree_query on the 2 x 3 product tree: 9 nodes, 6 paths, depth 2, and heads 1
    and 2 must supply their top-2 and top-3 (wiblog "Tree attention" worked example)."""
    tree = mb.Tree(synth.cartesian_choices((2, 3)))
    assert tree.query() == (9, 6, 2, [2, 3])


@pytest.mark.parametrize("name", ["tiny", "small_bf16"])
def test_rope_step_matches_oracle(mb, name, near_ties):
    """With rotary position encoding, the tree's q and k are turned at the position ids the
    tree expansion produced: attention outputs match the oracle's rotated pass, the rotated
    keys match apply_rope, the committed cache rows are the rotated keys, and the outputs
    differ from the unrotated pass (positions matter)."""
    wl = synth.WORKLOADS["tiny"] if name == "tiny" else SMALL_BF16
    kind = wl.dtype
    inp = synth.make_inputs(wl, "cuda", variant="plant", plant_depth=2 if name == "tiny" else None)
    step = make_step(mb, wl, inp, rope=True, rope_theta=10000.0)
    kc, vc, kl = inp.k_cache.clone(), inp.v_cache.clone(), inp.kv_len.clone()
    step.run(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, inp.X, inp.q, inp.k_new, inp.v_new, kc, vc, kl,
             0.7, wl.posterior_threshold, wl.posterior_alpha, root=inp.root)
    torch.cuda.synchronize()
    o = step_oracle_inputs(inp)
    tt = oracle.tree_tables(inp.choices)
    pos = npi(step.positions)
    _, pos_o = oracle.tree_tokens(tt, npi(step.root), npi(step.topk_ids), npi(inp.kv_len))
    assert np.array_equal(pos, pos_o)
    a_o = oracle.tree_attention(o["q"], o["k_new"], o["v_new"], o["k_cache"], o["v_cache"], npi(inp.kv_len), tt,
                                1.0 / math.sqrt(wl.D), positions=pos_o, rope_theta=10000.0)
    assert rel_err(step.attn_out, a_o) < TOL[kind]
    a_plain = oracle.tree_attention(o["q"], o["k_new"], o["v_new"], o["k_cache"], o["v_cache"], npi(inp.kv_len), tt,
                                    1.0 / math.sqrt(wl.D))
    assert rel_err(step.attn_out, a_plain) > 10 * TOL[kind]
    k_o = oracle.apply_rope(o["k_new"], pos_o, 10000.0)
    assert rel_err(step.k_rot, k_o) < (1e-5 if kind == "f32" else 1e-2)
    # the commit appended the rotated keys (bit-exact copies of k_rot) and the plain values
    kl0 = npi(inp.kv_len)
    for b in range(wl.B):
        best = int(step.best_node[b])
        chain = tt.ancestors[best] + [best]
        for d, node in enumerate(chain):
            assert torch.equal(kc[b, :, kl0[b] + d], step.k_rot[b, node])
            assert torch.equal(vc[b, :, kl0[b] + d], inp.v_new[b, node])
    near_ties(0)


# ----------------------------------------------------------------------------- tie-break variants

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_joint_probability_tie_break_hand_example(mb, dtype):
    """The hand-built 2 x 3 tree of the oracle's pin, fed through medusa_verify_accept (an
    identity lm_head, so each node's hidden state carries its logits): the first-in-order
    rule keeps node (0,0), the joint-probability rule node (1,2) with tokens 0, 2, 5."""
    tree = mb.Tree(synth.cartesian_choices((2, 3)))
    T, H, V = 9, 8, 6
    X = torch.zeros(1, T, H, dtype=torch.float64)
    X[0, 0, :6] = torch.log(torch.tensor([1, 3, 1, 1, 1, 1.0], dtype=torch.float64))
    X[0, 1, :6] = torch.log(torch.tensor([1, 1, 1, 2, 1, 1.0], dtype=torch.float64))
    X[0, 2, :6] = torch.log(torch.tensor([1, 1, 1, 1, 1, 40.0], dtype=torch.float64))
    X = X.to(dtype).cuda()
    lm = torch.zeros(V, H, dtype=dtype, device="cuda")
    lm[torch.arange(V), torch.arange(V)] = 1
    tokens = torch.tensor([[0, 1, 2, 3, 4, 5, 3, 4, 5]], dtype=torch.int32, device="cuda")
    dc = mb.MEDUSA_BF16 if dtype == torch.bfloat16 else mb.MEDUSA_F32
    ws = mb.workspace(mb.medusa_verify_accept_workspace_size(tree, 1, H, V, dc), "cuda")
    res = {}
    for rule in ("first", "joint"):
        out = [torch.full((1,), -1, dtype=torch.int32, device="cuda") for _ in range(4)]
        acc_tok = torch.full((1, 3), -9, dtype=torch.int32, device="cuda")
        mb.medusa_verify_accept(tree, X, lm, tokens, 1.0, 0.09, 0.3, out[0], out[1], out[2], acc_tok, out[3], ws,
                                tie_break=rule)
        torch.cuda.synchronize()
        res[rule] = (int(out[0]), int(out[2]), acc_tok[0].tolist())
    assert res["first"] == (2, 3, [0, 1, 3])
    assert res["joint"] == (2, 8, [0, 2, 5])


@pytest.mark.parametrize("temperature", [0.0, 0.7])
@pytest.mark.parametrize("wl", [SMALL_BF16, SMALL_BF16_D64], ids=lambda w: w.name)
def test_joint_tie_break_step(mb, wl, temperature, near_ties):
    """Whole step with the joint-probability tie-break against the oracle's (random inputs
    accept many equally deep nodes at temperature 0.7, so the rule decides)."""
    inp = synth.make_inputs(wl, "cuda")
    step, kc, vc, kl = run_step(mb, wl, inp, temperature, tie_break="joint")
    near = near_ties(check_full(wl, inp, step, kc, vc, kl, temperature, tie_break="joint"))
    assert near <= 3


@pytest.mark.parametrize("name", ["tiny", "small_bf16"])
def test_fused_commit_matches_separate_calls(mb, name):
    """medusa_verify_accept_commit (the commit run by the acceptance's CTA) leaves the same
    results, cache, kv_len and status as medusa_verify_accept followed by medusa_kv_commit,
    including a request whose accepted rows would pass Lmax (flagged, cache untouched)."""
    wl = SMALL_BF16 if name == "small_bf16" else synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda", variant="plant")
    kl_start = inp.kv_len.clone()
    kl_start[0] = wl.Lmax              # request 0 cannot take even its root row
    outs = []
    for fused in (False, True):
        step = make_step(mb, wl, inp)
        kc, vc, kl = inp.k_cache.clone(), inp.v_cache.clone(), kl_start.clone()
        step.root.copy_(inp.root)
        step.heads(inp.h, inp.W1, inp.b1, inp.W2)
        step.build(kl)
        step.attention(inp.q, inp.k_new, inp.v_new, kc, vc, kl)
        if fused:
            step.verify_commit(inp.X, inp.lm_head, inp.k_new, inp.v_new, kc, vc, kl, 0.7, wl.posterior_threshold,
                               wl.posterior_alpha)
        else:
            step.verify(inp.X, inp.lm_head, 0.7, wl.posterior_threshold, wl.posterior_alpha)
            step.commit(inp.k_new, inp.v_new, kc, vc, kl)
        torch.cuda.synchronize()
        outs.append((step.results.clone(), step.dev_status.clone(), kc, vc, kl))
    (r0, s0, kc0, vc0, kl0), (r1, s1, kc1, vc1, kl1) = outs
    assert torch.equal(r0, r1) and torch.equal(s0, s1)
    assert torch.equal(kl0, kl1) and torch.equal(kc0, kc1) and torch.equal(vc0, vc1)
    assert int(s1[0]) & mb.DEV_KV_OVERFLOW and int(kl1[0]) == wl.Lmax
    assert torch.equal(kc1[0], inp.k_cache[0])
    if wl.B > 1:
        assert all(int(kl1[b]) > int(kl_start[b]) for b in range(1, wl.B))
