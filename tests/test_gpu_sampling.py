"""GPU parity of the nucleus (top-p) draw of the next token (medusa_sample_next).

The draw u is an input (seeded), so the GPU and the oracle make the same
decision unless the oracle's margin (u times the nucleus mass against a
running-mass step, or top_p against the nucleus edge) is below the float
tolerance: such near-ties are counted and reported, not failed.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import DELTA, SMALL_BF16, np64, npi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mb():
    assert torch.cuda.is_available()
    import medusa_head_speculative_04_b300 as m
    return m


def test_nucleus_hand_example(mb):
    """q = (0.1, 0.2, 0.7), top_p 0.75: nucleus {1, 2}; u 0.2 -> 1, u 0.5 -> 2, u 0.99 -> 2;
    top_p 1 with u 0.05 -> token 0; temperature 0 -> token 2."""
    tree = mb.Tree([])
    logits = torch.log(torch.tensor([0.1, 0.2, 0.7], device="cuda")).view(1, 1, 3).repeat(5, 1, 1).contiguous()
    best = torch.zeros(5, dtype=torch.int32, device="cuda")
    u = torch.tensor([0.2, 0.5, 0.99, 0.05, 0.3], device="cuda")
    out = torch.full((5,), -1, dtype=torch.int32, device="cuda")
    mb.medusa_sample_next(tree, logits, best, u, 1.0, 0.75, out)
    torch.cuda.synchronize()
    assert out[:3].tolist() == [1, 2, 2]
    mb.medusa_sample_next(tree, logits, best, u, 1.0, 1.0, out)
    torch.cuda.synchronize()
    assert int(out[3]) == 0
    mb.medusa_sample_next(tree, logits, best, u, 0.0, 0.75, out)
    torch.cuda.synchronize()
    assert out.tolist() == [2] * 5


@pytest.mark.parametrize("name", ["small_bf16", "vicuna7b"])
@pytest.mark.parametrize("top_p", [0.5, 0.9, 1.0])
def test_nucleus_next_token_matches_oracle(mb, name, top_p, near_ties):
    wl = SMALL_BF16 if name == "small_bf16" else synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda")
    step = mb.MedusaStep(inp.choices, wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.k_needed(),
                         inp.dtype, keep_logits=True)
    kc, vc, kl = inp.k_cache.clone(), inp.v_cache.clone(), inp.kv_len.clone()
    step.run(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, inp.X, inp.q, inp.k_new, inp.v_new, kc, vc, kl, 0.7,
             root=inp.root)
    rng = synth.SplitMix64(synth.tensor_seed(wl.config_id, 0x55))
    draws = [(rng.next() >> 11) / float(1 << 53) for _ in range(4 * wl.B)]
    near = 0
    for rep in range(4):
        u = torch.tensor(draws[rep * wl.B:(rep + 1) * wl.B], dtype=torch.float32, device="cuda")
        out = torch.full((wl.B,), -1, dtype=torch.int32, device="cuda")
        mb.medusa_sample_next(step.tree, step.logits, step.best_node, u, 0.7, top_p, out)
        torch.cuda.synchronize()
        best = npi(step.best_node)
        for b in range(wl.B):
            z_o = np64(inp.X[b, best[b]]) @ np64(inp.lm_head).T
            r = oracle.nucleus_next(z_o, 0.7, top_p, float(u[b]))
            if int(out[b]) != r["token"]:
                assert r["margin"] < DELTA[wl.dtype] * 10, (b, int(out[b]), r)
                near += 1
    assert near_ties(near) <= 2


def test_nucleus_limits_on_gpu(mb):
    """A tiny top_p keeps only the greedy token (for every draw), which then equals the
    verification's next root."""
    wl = SMALL_BF16
    inp = synth.make_inputs(wl, "cuda", variant="plant")
    step = mb.MedusaStep(inp.choices, wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.k_needed(),
                         inp.dtype, keep_logits=True)
    kc, vc, kl = inp.k_cache.clone(), inp.v_cache.clone(), inp.kv_len.clone()
    step.run(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, inp.X, inp.q, inp.k_new, inp.v_new, kc, vc, kl, 0.7,
             root=inp.root)
    out = torch.full((wl.B,), -1, dtype=torch.int32, device="cuda")
    for uval in (0.0, 0.5, 0.999):
        u = torch.full((wl.B,), uval, device="cuda")
        mb.medusa_sample_next(step.tree, step.logits, step.best_node, u, 0.7, 1e-6, out)
        torch.cuda.synchronize()
        assert torch.equal(out, step.next_root)
