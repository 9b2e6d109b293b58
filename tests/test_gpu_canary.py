"""Every output of a step stays inside its buffer.

Each output tensor of a whole step (and the KV cache the commit writes) is a
view into a larger buffer whose guard regions before and after the view hold a
fixed bit pattern; after the step, and after a second step through the captured
CUDA graph, every guard word must still hold it.  The step's results are also
compared with those of the same step on plain buffers, so the guarded run takes
the same paths.  Workloads: the fp32 tiny step, a bf16 batch of three (tensor-core
heads), the 7B shape with the next step's heads on the accepted rows.
"""
import pytest
import torch

import synth
from _util import SMALL_BF16

pytestmark = pytest.mark.gpu

PAD = 256  # guard elements on each side (1 KB for 4-byte types): keeps 16-byte alignment
PATTERN = {torch.float32: 0x7FC00ABC, torch.int32: 0x5A5A5A5A, torch.bfloat16: 0x7FAB}
OUTPUTS = ("topk_ids", "topk_vals", "root", "tokens", "positions", "candidates", "attn_out", "dev_status",
           "head_logits", "logits", "node_p", "node_H")
RESULTS = ("accept_len", "best_path", "best_node", "next_root", "accepted_tokens")


@pytest.fixture(scope="module")
def mb():
    assert torch.cuda.is_available(), "the CUDA parity tests need a GPU"
    import medusa_head_speculative_04_b300 as m
    return m


class Guarded:
    """A view of `like`'s shape and dtype inside a buffer with guard regions."""

    def __init__(self, like: torch.Tensor):
        n = like.numel()
        self.buf = torch.empty(n + 2 * PAD, dtype=like.dtype, device=like.device)
        bits = self.buf.view(torch.int16 if like.dtype == torch.bfloat16 else torch.int32)
        pat = PATTERN[like.dtype]
        bits.fill_(pat - (1 << 16) if like.dtype == torch.bfloat16 and pat >= 1 << 15 else pat)
        self.view = self.buf[PAD:PAD + n].view(like.shape)
        self.view.copy_(like)
        self.n = n

    def intact(self) -> bool:
        bits = self.buf.view(torch.int16 if self.buf.dtype == torch.bfloat16 else torch.int32)
        pat = PATTERN[self.buf.dtype]
        want = pat - (1 << 16) if self.buf.dtype == torch.bfloat16 and pat >= 1 << 15 else pat
        return bool((bits[:PAD] == want).all()) and bool((bits[PAD + self.n:] == want).all())


def guard_step(step):
    """Swap the step's output tensors for guarded views; the results buffer is split
    into guarded per-field views (each read by its own pointer)."""
    guards = {}
    for name in OUTPUTS + RESULTS:
        t = getattr(step, name)
        if t is None:
            continue
        g = Guarded(t.contiguous())
        setattr(step, name, g.view)
        guards[name] = g
    return guards


def run(mb, wl, inp, guarded: bool, tau: float):
    step = mb.MedusaStep(inp.choices, wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.k_needed(),
                         inp.dtype, keep_head_logits=True, keep_logits=True,
                         kv_len_hint=max(wl.kv_lens()))
    guards = guard_step(step) if guarded else {}
    if guarded:
        gk, gv = Guarded(inp.k_cache), Guarded(inp.v_cache)
        kc, vc = gk.view, gv.view
        guards["k_cache"], guards["v_cache"] = gk, gv
    else:
        kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    kl = inp.kv_len.clone()
    step.run(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, inp.X, inp.q, inp.k_new, inp.v_new, kc, vc, kl, tau,
             wl.posterior_threshold, wl.posterior_alpha, root=inp.root)
    step.heads_from_tree(inp.X, inp.W1, inp.b1, inp.W2)
    torch.cuda.synchronize()
    return step, guards, kc, vc, kl


@pytest.mark.parametrize("name", ["tiny", "small_bf16", "vicuna7b"])
def test_outputs_stay_inside_their_buffers(mb, name):
    wl = SMALL_BF16 if name == "small_bf16" else synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda", variant="plant")
    plain, _, kc0, vc0, kl0 = run(mb, wl, inp, False, 0.7)
    step, guards, kc, vc, kl = run(mb, wl, inp, True, 0.7)
    bad = [n for n, g in guards.items() if not g.intact()]
    assert not bad, bad
    for name_ in ("topk_ids", "root", "tokens", "positions", "candidates", "accept_len", "best_node", "next_root",
                  "accepted_tokens", "dev_status"):
        assert torch.equal(getattr(step, name_), getattr(plain, name_)), name_
    assert torch.equal(kl, kl0) and torch.equal(kc, kc0) and torch.equal(vc, vc0)
    # a second step through the captured graph on the same guarded buffers
    kl.copy_(inp.kv_len)
    g = step.capture(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, inp.X, inp.q, inp.k_new, inp.v_new, kc, vc, kl,
                     0.7, wl.posterior_threshold, wl.posterior_alpha, root=inp.root)
    g.replay()
    torch.cuda.synchronize()
    bad = [n for n, gd in guards.items() if not gd.intact()]
    assert not bad, bad
