"""GPU parity of the heads on the tree nodes' hidden states
(medusa_heads_topk_tree): the next step's candidates taken from the
verification pass's hidden states.

wiblog.cn "Medusa multi-head speculative decoding", section "Inference flow in
an online chat service": the verification pass that scores the candidates also
yields the next round's candidates, with no extra forward pass.  The kernels
gather each request's accepted row and run the heads on those rows (bf16 from
three requests: tensor-core GEMMs); the oracle runs the heads on the tree rows
and keeps the accepted one.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from _full import check_commit, check_verify_accept
from _util import DELTA, SMALL_BF16, TOL, check_topk, np64, npi, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mb():
    assert torch.cuda.is_available()
    import medusa_head_speculative_04_b300 as m
    return m


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def tree_heads_oracle(wl, X, best, inp):
    """Per-head oracle logits [B, K, V] of the accepted rows (heads one at a time)."""
    return np.concatenate([oracle.tree_heads(_f64(X), best, _f64(inp.W1[k:k + 1]), _f64(inp.b1[k:k + 1]),
                                             _f64(inp.W2[k:k + 1]), u_bf16=(wl.dtype == "bf16"))[1]
                           for k in range(wl.K)], axis=1)


@pytest.mark.parametrize("keep_logits", [True, False])
@pytest.mark.parametrize("name", ["tiny", "small_bf16", "vicuna7b"])
def test_tree_heads_match_oracle(mb, name, keep_logits, near_ties):
    wl = SMALL_BF16 if name == "small_bf16" else synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda")
    tt = oracle.tree_tables(inp.choices)
    best = np.array([(5 * b + 3) % tt.T for b in range(wl.B)])   # any node of each request
    tree = mb.Tree(inp.choices)
    k = wl.k_needed()
    dc = mb.MEDUSA_BF16 if inp.dtype == torch.bfloat16 else mb.MEDUSA_F32
    ws = mb.workspace(mb.medusa_heads_topk_tree_workspace_size(tree, wl.B, wl.H, wl.V, wl.K, k, dc), "cuda")
    ids = torch.full((wl.B, wl.K, k), -3, dtype=torch.int32, device="cuda")
    vals = torch.zeros(wl.B, wl.K, k, device="cuda")
    logits = torch.zeros(wl.B, wl.K, wl.V, device="cuda") if keep_logits else None
    best_d = torch.tensor(best, dtype=torch.int32, device="cuda")
    for call in range(2):   # the workspace's counters reset themselves
        ids.fill_(-3)
        mb.medusa_heads_topk_tree(tree, inp.X, inp.W1, inp.b1, inp.W2, best_d, k, ids, vals, ws, head_logits=logits)
        torch.cuda.synchronize()
        z_o = tree_heads_oracle(wl, inp.X, best, inp)
        if keep_logits:
            assert rel_err(logits, z_o) < TOL[wl.dtype], call
        near = check_topk(ids, vals, z_o, k, DELTA[wl.dtype])
        assert rel_err(vals, np.take_along_axis(z_o, npi(ids), axis=-1)) < TOL[wl.dtype]
    assert near_ties(near) <= 2


def test_tree_heads_zero_init_follow_the_verification(mb, near_ties):
    """Heads in their start state (W1 = b1 = 0, W2_k = lm_head): the logits the heads give
    on the accepted row match that row's verification logits, so every head's top-1 is the
    verification pass's next root."""
    wl = SMALL_BF16
    inp = synth.make_inputs(wl, "cuda", variant="zeroinit")
    step = mb.MedusaStep(inp.choices, wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.k_needed(),
                         inp.dtype, keep_head_logits=True, keep_logits=True)
    kc, vc, kl = inp.k_cache.clone(), inp.v_cache.clone(), inp.kv_len.clone()
    step.run(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, inp.X, inp.q, inp.k_new, inp.v_new, kc, vc, kl, 0.7,
             root=inp.root)
    step.heads_from_tree(inp.X, inp.W1, inp.b1, inp.W2)
    torch.cuda.synchronize()
    best = npi(step.best_node)
    zv = np64(step.logits)[np.arange(wl.B), best]
    near = 0
    for b in range(wl.B):
        for kk in range(wl.K):
            assert rel_err(step.head_logits[b, kk], zv[b]) < TOL[wl.dtype]
            top = int(step.topk_ids[b, kk, 0])
            if top != int(step.next_root[b]):
                srt = np.sort(zv[b])
                assert srt[-1] - srt[-2] < DELTA[wl.dtype] * max(1.0, abs(srt[-1]))
                near += 1
    assert int(step.root[0]) == int(step.next_root[0])
    assert near_ties(near) <= 1


@pytest.mark.parametrize("name", ["small_bf16", "vicuna7b"])
def test_two_step_loop_continues_from_the_accepted_row(mb, name, near_ties):
    """Step 1 runs the whole step; the heads over its tree states give the candidates of
    step 2, which then expands, attends, verifies (new tree states) and commits.  Step 2's
    tree tokens, acceptance and commit match the oracle run on the accepted row of step 1."""
    wl = SMALL_BF16 if name == "small_bf16" else synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda", variant="plant")
    step = mb.MedusaStep(inp.choices, wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.k_needed(),
                         inp.dtype, kv_len_hint=max(wl.kv_lens()), keep_node_stats=False)
    kc, vc, kl = inp.k_cache.clone(), inp.v_cache.clone(), inp.kv_len.clone()
    step.run(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, inp.X, inp.q, inp.k_new, inp.v_new, kc, vc, kl, 0.7,
             wl.posterior_threshold, wl.posterior_alpha, root=inp.root)
    step.heads_from_tree(inp.X, inp.W1, inp.b1, inp.W2)
    torch.cuda.synchronize()
    best1, root2, kv2 = npi(step.best_node), npi(step.next_root), kl.clone()
    cache2_k, cache2_v = kc.clone(), vc.clone()
    # oracle: candidates of step 2 from step 1's accepted rows
    k = wl.k_needed()
    z_o = tree_heads_oracle(wl, inp.X, best1, inp)
    near = check_topk(step.topk_ids, step.topk_vals, z_o, k, DELTA[wl.dtype])
    # step 2 on new activations, continuing from the committed cache
    nxt = synth.make_inputs(dataclasses.replace(wl, config_id=wl.config_id + 60), "cuda", with_weights=False)
    step.build(kl)
    step.attention(nxt.q, nxt.k_new, nxt.v_new, kc, vc, kl)
    step.verify(nxt.X, inp.lm_head, 0.7, wl.posterior_threshold, wl.posterior_alpha)
    step.commit(nxt.k_new, nxt.v_new, kc, vc, kl)
    torch.cuda.synchronize()
    tt = oracle.tree_tables(inp.choices)
    tok_o, pos_o = oracle.tree_tokens(tt, root2, npi(step.topk_ids), npi(kv2))
    assert np.array_equal(npi(step.tokens), tok_o) and np.array_equal(npi(step.positions), pos_o)
    step2 = dataclasses.replace(inp, X=nxt.X, q=nxt.q, k_new=nxt.k_new, v_new=nxt.v_new, k_cache=cache2_k,
                                v_cache=cache2_v, kv_len=kv2, plant=None)
    near += check_verify_accept(wl, step2, step, tt, 0.7)
    check_commit(wl, step2, step, kc, vc, kl, tt)
    assert near_ties(near) <= 3
