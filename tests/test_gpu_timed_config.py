"""GPU parity of the configuration the benchmark times.

bench.py runs the step keeping nothing beyond the per-request results: no head
logits, no verification logits, no node statistics, the cache split sized from
the workload's kv_len hint, the whole step captured in a CUDA graph and
replayed.  That takes branches of its own: the tensor-core heads write their
logits into the workspace, the verification epilogue writes no logits, the fp32
verification writes into a workspace buffer, and the merge writes no node
statistics.  These tests run exactly that configuration, replay the captured
graph twice with different activations (a planted accept path, then unrelated
random rows), and compare every discrete output, the next root and the
committed cache with the oracle (near-ties counted and reported).
"""
import dataclasses

import pytest
import torch

import oracle
import synth
from _full import check_commit, check_heads, check_tree, check_verify_accept
from _util import SMALL_BF16

pytestmark = pytest.mark.gpu

ACTIVATIONS = ("h", "X", "q", "k_new", "v_new", "root")   # refilled before each replay


@pytest.fixture(scope="module")
def mb():
    assert torch.cuda.is_available(), "the CUDA parity tests need a GPU"
    import medusa_head_speculative_04_b300 as m
    return m


def timed_step(mb, wl, inp, temperature):
    """The benchmark's step object and its captured graph (bench.py builds the same).

    Every tensor the graph reads must outlive it, the source of the prologue's kv_len
    reset included: it is returned with the rest (a freed source block could be handed
    to the next allocation and the replay would copy whatever that holds)."""
    step = mb.MedusaStep(inp.choices, wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.k_needed(),
                         inp.dtype, kv_len_hint=max(wl.kv_lens()), keep_node_stats=False)
    assert step.head_logits is None and step.logits is None and step.node_p is None
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    kl0 = inp.kv_len.clone()
    kl = kl0.clone()
    act = {k: getattr(inp, k).clone() for k in ACTIVATIONS}
    g = step.capture(act["h"], inp.W1, inp.b1, inp.W2, inp.lm_head, act["X"], act["q"], act["k_new"],
                     act["v_new"], kc, vc, kl, temperature, wl.posterior_threshold, wl.posterior_alpha,
                     root=act["root"], prologue=lambda: kl.copy_(kl0))
    act["kv_len0"] = kl0
    return step, g, act, kc, vc, kl


def replay_and_check(wl, inp, step, g, act, kc, vc, kl, temperature, src):
    """Refill the captured activations from ``src``, replay, compare with the oracle."""
    for k in ACTIVATIONS:
        act[k].copy_(getattr(src, k))
    kc.copy_(inp.k_cache)
    vc.copy_(inp.v_cache)
    for t in (step.results, step.dev_status, step.topk_ids, step.tokens):
        t.fill_(-5)
    step.dev_status.zero_()
    g.replay()
    torch.cuda.synchronize()
    cur = dataclasses.replace(inp, **{k: getattr(src, k) for k in ACTIVATIONS},
                              plant=src.plant if src is inp else None)
    tt = oracle.tree_tables(inp.choices)
    near = check_heads(wl, cur, step)
    check_tree(wl, cur, step, tt)
    near += check_verify_accept(wl, cur, step, tt, temperature)
    check_commit(wl, cur, step, kc, vc, kl, tt)
    assert int((step.dev_status & ~1).max()) == 0, step.dev_status
    if cur.plant is not None:
        assert all(int(step.accept_len[b]) >= cur.plant["depths"][b] for b in range(wl.B))
    return near


def other_activations(wl, dev):
    """Unrelated random activations of the same shapes (the weights stay the captured ones)."""
    return synth.make_inputs(dataclasses.replace(wl, config_id=wl.config_id + 40), dev, with_weights=False)


# tiny: fp32 verification into the workspace buffer; small_bf16 (B = 3): tensor-core heads
# writing their logits into the workspace; vicuna7b: the benchmark's own workload
CASES = [("tiny", 0.0), ("tiny", 0.7), ("small_bf16", 0.7), ("small_bf16", 0.0), ("vicuna7b", 0.7),
         ("vicuna7b", 0.0)]


@pytest.mark.parametrize("name,temperature", CASES)
def test_timed_config_matches_oracle(mb, name, temperature, near_ties):
    wl = SMALL_BF16 if name == "small_bf16" else synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda", variant="plant", plant_depth=2 if name == "tiny" else None)
    step, g, act, kc, vc, kl = timed_step(mb, wl, inp, temperature)
    near = replay_and_check(wl, inp, step, g, act, kc, vc, kl, temperature, inp)
    near += replay_and_check(wl, inp, step, g, act, kc, vc, kl, temperature, other_activations(wl, "cuda"))
    assert near_ties(near) <= 4


@pytest.mark.slow
def test_timed_config_llama8b_b16(mb, near_ties):
    """Batch 16 at the Llama-3.1-8B shape: both head GEMMs on the tensor cores with the
    logits in the workspace, and the compute-bound lm_head GEMM over 1040 tree rows."""
    wl = synth.WORKLOADS["llama8b_b16"]
    inp = synth.make_inputs(wl, "cuda", variant="plant")
    step, g, act, kc, vc, kl = timed_step(mb, wl, inp, 0.7)
    near = replay_and_check(wl, inp, step, g, act, kc, vc, kl, 0.7, inp)
    assert near_ties(near) <= 4
