"""The allocation-free heads entry point against the oracle and against the
workspace entry point.

medusa_heads_topk_noalloc exists for callers that must not allocate device
memory (cudaMalloc can synchronise the device and take a driver-wide lock, so a
latency-bound decode loop or a plugin living in another framework's memory
pool may not call it).  Its scratch is a fixed array inside the library that
every call shares, so each test calls it twice in a row: the second call must
not be disturbed by what the first left in that array.  This file is collected
last on purpose, so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import DELTA, TOL, check_topk, np64, npi, rel_err

NOALLOC_BYTES = 8 << 20   # MEDUSA_NOALLOC_SCRATCH_BYTES


def _outs(B, K, k, V, dev):
    return (torch.full((B, K, k), -7, dtype=torch.int32, device=dev),
            torch.zeros(B, K, k, dtype=torch.float32, device=dev),
            torch.full((B,), -7, dtype=torch.int32, device=dev),
            torch.zeros(B, K, V, dtype=torch.float32, device=dev))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(mb, inp, lm, B, H, V, K, k, dc, outs):
    ids, vals, root, logits = outs
    return mb.lib.medusa_heads_topk_noalloc(
        _p(inp.h), _p(inp.W1), _p(inp.b1), _p(inp.W2), _p(lm), B, H, V, K, k, dc, _p(logits), _p(ids), _p(vals),
        _p(root), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


WORKLOADS = {
    "tiny": synth.WORKLOADS["tiny"],
    # bf16 at batch 3 with the root given: the workspace entry point takes the tensor-core
    # path here, the allocation-free one the CUDA-core path
    "bf16_b3": synth.Workload("noalloc_bf16", 31, H=512, V=3001, K=3, Hq=8, Hkv=2, D=128, L=64, B=3,
                              dtype="bf16", tree=("cartesian", (3, 2, 2))),
    "llama8b_b4": synth.WORKLOADS["llama8b_b4"],
}


@pytest.mark.gpu
@pytest.mark.parametrize("name,with_lm", [("tiny", True), ("bf16_b3", False), ("bf16_b3", True),
                                          ("llama8b_b4", True)])
def test_noalloc_matches_oracle_and_workspace_entry_point(name, with_lm, near_ties):
    assert torch.cuda.is_available()
    import medusa_head_speculative_04_b300 as mb
    wl = WORKLOADS[name]
    dev = torch.device("cuda", 0)
    inp = synth.make_inputs(wl, dev, variant="plant")
    B, H, V, K, k = wl.B, wl.H, wl.V, wl.K, wl.k_needed()
    dc = mb.MEDUSA_BF16 if inp.dtype == torch.bfloat16 else mb.MEDUSA_F32
    lm = inp.lm_head if with_lm else None
    tol, delta = TOL[wl.dtype], DELTA[wl.dtype]

    # the oracle: head logits, their top-k, and the root when lm_head is given
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    z_o = np.concatenate([oracle.medusa_heads(f64(inp.h), f64(inp.W1[i:i + 1]), f64(inp.b1[i:i + 1]),
                                              f64(inp.W2[i:i + 1]), u_bf16=(wl.dtype == "bf16"))[1]
                          for i in range(K)], axis=1)
    root_o = oracle.base_root(f64(inp.h), f64(inp.lm_head)) if with_lm else None
    z_root = f64(inp.h) @ f64(inp.lm_head).T if with_lm else None

    # the workspace entry point on the same inputs
    ids_r, vals_r, root_r, log_r = _outs(B, K, k, V, dev)
    ws = mb.workspace(mb.medusa_heads_topk_workspace_size(B, H, V, K, k, with_lm, dc), dev)
    mb.medusa_heads_topk(inp.h, inp.W1, inp.b1, inp.W2, lm, k, ids_r, vals_r, root_r, ws, head_logits=log_r)
    torch.cuda.synchronize()

    near = 0
    for call in range(2):
        outs = _outs(B, K, k, V, dev)
        ids, vals, root, logits = outs
        rc = _noalloc(mb, inp, lm, B, H, V, K, k, dc, outs)
        assert rc == 0, mb.lib.medusa_status_string(rc)
        torch.cuda.synchronize()
        # against the oracle
        assert rel_err(logits, z_o) < tol, call
        near += check_topk(ids, vals, z_o, k, delta)
        assert rel_err(vals, np.take_along_axis(z_o, npi(ids), axis=-1)) < tol, call
        if with_lm:
            for b in range(B):
                g, r = int(root[b]), int(root_o[b])
                if g != r:
                    assert abs(z_root[b, g] - z_root[b, r]) < delta * max(1.0, abs(z_root[b, r])), (call, b)
                    near += 1
        else:
            assert torch.equal(root, torch.full_like(root, -7)), "root_tok is an input when lm_head is NULL"
        # against the workspace entry point: ids equal except at counted near-ties
        for r, (a, c) in enumerate(zip(npi(ids).reshape(-1, k), npi(ids_r).reshape(-1, k))):
            for t in np.nonzero(a != c)[0]:
                zr = z_o.reshape(-1, V)[r]
                assert abs(zr[a[t]] - zr[c[t]]) < delta * max(1.0, abs(zr[c[t]])), (call, r, t)
        assert rel_err(logits, np64(log_r)) < tol, call
        assert rel_err(vals, np64(vals_r)) < tol, call
    assert near_ties(near) <= 2


def _fp32_need(mb, B, H, V, K, k):
    # fp32 always plans the CUDA-core path, so the workspace size is the scratch need
    return mb.lib.medusa_heads_topk_workspace_size(B, H, V, K, k, 0, mb.MEDUSA_F32)


def _boundary_shape(mb):
    """An fp32 shape whose scratch need is at most the array's size, and the next hidden
    size up (a multiple of 8), whose need is above it.  Batch 64 with top-48 keeps the
    per-CTA candidate lists large, so the boundary falls at a small hidden size."""
    B, V, K, k = 64, 4096, 5, 48
    H = 8
    assert 0 < _fp32_need(mb, B, H, V, K, k) <= NOALLOC_BYTES
    while _fp32_need(mb, B, H + 8, V, K, k) <= NOALLOC_BYTES:
        H += 8
        assert H < 4096
    assert _fp32_need(mb, B, H, V, K, k) <= NOALLOC_BYTES < _fp32_need(mb, B, H + 8, V, K, k)
    return B, H, V, K, k


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import medusa_head_speculative_04_b300 as mb
    p = 0x10000  # aligned fake addresses: the call must fail before touching them
    # batch 64 x 5 heads x hidden 16384 in fp32 needs ~21 MB of u alone > the 8 MiB array
    rc = mb.lib.medusa_heads_topk_noalloc(p, p, p, p, None, 64, 16384, 1000, 5, 4, mb.MEDUSA_F32, None, p, p, p,
                                          None)
    assert rc == -6
    assert b"scratch" in mb.lib.medusa_status_string(rc)
    # one hidden-size step past the largest shape that fits is rejected too
    B, H, V, K, k = _boundary_shape(mb)
    rc = mb.lib.medusa_heads_topk_noalloc(p, p, p, p, None, B, H + 8, V, K, k, mb.MEDUSA_F32, None, p, p, p, None)
    assert rc == -6


@pytest.mark.gpu
def test_noalloc_runs_at_its_largest_shape():
    """The largest fp32 shape that fits the array runs (twice) and matches the oracle."""
    import medusa_head_speculative_04_b300 as mb
    B, H, V, K, k = _boundary_shape(mb)
    wl = synth.Workload("noalloc_edge", 32, H=H, V=V, K=K, Hq=4, Hkv=4, D=64, L=8, B=B, dtype="f32",
                        tree=("cartesian", (2,)), topk=k)
    dev = torch.device("cuda", 0)
    inp = synth.make_inputs(wl, dev)
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    _, z_o = oracle.medusa_heads(f64(inp.h), f64(inp.W1), f64(inp.b1), f64(inp.W2), u_bf16=False)
    for call in range(2):
        outs = _outs(B, K, k, V, dev)
        rc = _noalloc(mb, inp, None, B, H, V, K, k, mb.MEDUSA_F32, outs)
        assert rc == 0, mb.lib.medusa_status_string(rc)
        torch.cuda.synchronize()
        assert rel_err(outs[3], z_o) < TOL["f32"], call
        check_topk(outs[0], outs[1], z_o, k, DELTA["f32"])
