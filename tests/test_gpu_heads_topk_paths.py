"""GPU parity of the batched (tensor-core) heads over both of their top-k paths.

At B >= 3 in bf16 both head products run as tcgen05 GEMMs.  With k <= 16 the
W2 GEMM's epilogue keeps the top-k of every vocabulary tile in registers and a
second launch merges the tiles' candidates per (row, head); with k > 16 the
GEMM writes the logits and a selection pass reads them back.  Ultralytics
glossary "Medusa Heads", "How the heads predict the next tokens" (the head
function) and wiblog.cn "Medusa multi-head speculative decoding", "Medusa
decoding heads" (each head's top-k).  Every case is compared with the oracle,
with and without the caller keeping the head logits, on vocabularies whose last
tile is ragged; a row of NaN logits gets no candidate.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import DELTA, SMALL_BF16, TOL, check_topk, npi, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mb():
    assert torch.cuda.is_available(), "the CUDA parity tests need a GPU"
    import medusa_head_speculative_04_b300 as m
    return m


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run_heads(mb, inp, wl, topk, keep_logits):
    B, K, V = wl.B, wl.K, wl.V
    ws = mb.workspace(mb.medusa_heads_topk_workspace_size(B, wl.H, V, K, topk, 0, mb.MEDUSA_BF16), "cuda")
    ids = torch.full((B, K, topk), -3, dtype=torch.int32, device="cuda")
    vals = torch.zeros(B, K, topk, device="cuda")
    root = torch.zeros(B, dtype=torch.int32, device="cuda")
    logits = torch.zeros(B, K, V, device="cuda") if keep_logits else None
    for _ in range(2):   # a second call on the same workspace
        ids.fill_(-3)
        mb.medusa_heads_topk(inp.h, inp.W1, inp.b1, inp.W2, None, topk, ids, vals, root, ws, head_logits=logits)
    torch.cuda.synchronize()
    return ids, vals, logits


def oracle_logits(inp, wl):
    h = _f64(inp.h)
    return np.stack([oracle.medusa_heads(h, _f64(inp.W1[k:k + 1]), _f64(inp.b1[k:k + 1]), _f64(inp.W2[k:k + 1]),
                                         u_bf16=True)[1][:, 0] for k in range(wl.K)], axis=1)


@pytest.mark.parametrize("keep_logits", [False, True])
@pytest.mark.parametrize("topk", [1, 7, 16, 17, 40])
@pytest.mark.parametrize("V", [3001, 4101])
def test_batched_heads_topk_paths(mb, V, topk, keep_logits, near_ties):
    wl = dataclasses.replace(SMALL_BF16, name=f"heads_v{V}", config_id=70 + V % 7, V=V, B=5, K=4)
    inp = synth.make_inputs(wl, "cuda")
    ids, vals, logits = run_heads(mb, inp, wl, topk, keep_logits)
    z_o = oracle_logits(inp, wl)
    if keep_logits:
        assert rel_err(logits, z_o) < TOL["bf16"]
    near = check_topk(ids, vals, z_o, topk, DELTA["bf16"])
    assert rel_err(vals, np.take_along_axis(z_o, npi(ids), axis=-1)) < TOL["bf16"]
    assert near_ties(near) <= 3


@pytest.mark.parametrize("topk", [5, 20])
def test_batched_heads_nan_row_gets_no_candidate(mb, topk):
    """A NaN in one request's hidden state makes all its logits NaN: its entries are
    (-1, -inf) on both paths, and the other requests' top-k are those of the clean run."""
    wl = dataclasses.replace(SMALL_BF16, name="heads_nan", config_id=77, B=4)
    inp = synth.make_inputs(wl, "cuda")
    clean_ids, clean_vals, _ = run_heads(mb, inp, wl, topk, False)
    h = inp.h.clone()
    h[2, 11] = float("nan")
    ids, vals, _ = run_heads(mb, dataclasses.replace(inp, h=h), wl, topk, False)
    assert (ids[2] == -1).all() and torch.isneginf(vals[2]).all()
    keep = [0, 1, 3]
    assert torch.equal(ids[keep], clean_ids[keep]) and torch.equal(vals[keep], clean_vals[keep])


@pytest.mark.parametrize("with_lm", [False, True])
@pytest.mark.parametrize("B", [1, 2])
def test_vocabulary_stream_dynamic_split(mb, B, with_lm, near_ties):
    """One or two activation rows on a vocabulary long enough for the dynamic row split
    (at least 16 rows per warp) and not a multiple of the 4 rows a warp takes at a time,
    with and without the lm_head root block: top-k, head logits and root against the
    oracle."""
    wl = dataclasses.replace(SMALL_BF16, name="heads_dyn", config_id=78, V=7557, B=B, K=5)
    inp = synth.make_inputs(wl, "cuda")
    k = 10
    ws = mb.workspace(mb.medusa_heads_topk_workspace_size(B, wl.H, wl.V, wl.K, k, int(with_lm), mb.MEDUSA_BF16),
                      "cuda")
    ids = torch.full((B, wl.K, k), -3, dtype=torch.int32, device="cuda")
    vals = torch.zeros(B, wl.K, k, device="cuda")
    root = torch.full((B,), -3, dtype=torch.int32, device="cuda")
    logits = torch.zeros(B, wl.K, wl.V, device="cuda")
    for _ in range(2):   # the counters reset themselves
        mb.medusa_heads_topk(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head if with_lm else None, k, ids, vals, root,
                             ws, head_logits=logits)
    torch.cuda.synchronize()
    z_o = oracle_logits(inp, wl)
    assert rel_err(logits, z_o) < TOL["bf16"]
    near = check_topk(ids, vals, z_o, k, DELTA["bf16"])
    if with_lm:
        h, lm = _f64(inp.h), _f64(inp.lm_head)
        z_root = h @ lm.T
        for b in range(B):
            g, r = int(root[b]), int(oracle.base_root(h[b:b + 1], lm)[0])
            if g != r:
                assert abs(z_root[b, g] - z_root[b, r]) < DELTA["bf16"] * max(1.0, abs(z_root[b, r]))
                near += 1
    assert near_ties(near) <= 3
