"""The allocation-free heads entry point gives the same results as the
workspace one.

medusa_heads_topk_noalloc exists for callers that must not allocate device
memory (cudaMalloc can synchronise the device and take a driver-wide lock, so a
latency-bound decode loop or a plugin living in another framework's memory
pool may not call it).  Its scratch is a fixed array inside the library that
every call shares, so the test calls it twice in a row: the second call must
not be disturbed by what the first left in that array.  This file is collected
last on purpose.
"""
import ctypes

import pytest
import torch

import synth
from _util import TOL, rel_err

pytestmark = pytest.mark.gpu


def _outs(B, K, k, V, dev):
    return (torch.full((B, K, k), -7, dtype=torch.int32, device=dev),
            torch.zeros(B, K, k, dtype=torch.float32, device=dev),
            torch.full((B,), -7, dtype=torch.int32, device=dev),
            torch.zeros(B, K, V, dtype=torch.float32, device=dev))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("name", ["tiny", "small_bf16", "llama8b_b4"])
def test_noalloc_matches_workspace_entry_point(name):
    assert torch.cuda.is_available()
    import medusa_head_speculative_04_b300 as mb
    if name == "small_bf16":
        wl = synth.Workload("noalloc_bf16", 31, H=512, V=3001, K=3, Hq=8, Hkv=2, D=128, L=64, B=3,
                            dtype="bf16", tree=("cartesian", (3, 2, 2)))
    else:
        wl = synth.WORKLOADS[name]
    dev = torch.device("cuda", 0)
    inp = synth.make_inputs(wl, dev, variant="plant")
    B, H, V, K, k = wl.B, wl.H, wl.V, wl.K, wl.k_needed()
    dc = mb.MEDUSA_BF16 if inp.dtype == torch.bfloat16 else mb.MEDUSA_F32

    # reference: the workspace entry point
    ids_r, vals_r, root_r, log_r = _outs(B, K, k, V, dev)
    ws = mb.workspace(mb.medusa_heads_topk_workspace_size(B, H, V, K, k, True, dc), dev)
    mb.medusa_heads_topk(inp.h, inp.W1, inp.b1, inp.W2, inp.lm_head, k, ids_r, vals_r, root_r, ws,
                         head_logits=log_r)
    torch.cuda.synchronize()

    for call in range(2):
        ids, vals, root, logits = _outs(B, K, k, V, dev)
        rc = mb.lib.medusa_heads_topk_noalloc(
            _p(inp.h), _p(inp.W1), _p(inp.b1), _p(inp.W2), _p(inp.lm_head), B, H, V, K, k, dc, _p(logits),
            _p(ids), _p(vals), _p(root), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, mb.lib.medusa_status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_r), call
        assert torch.equal(root, root_r), call
        assert rel_err(vals, vals_r) < TOL[wl.dtype], call
        assert rel_err(logits, log_r) < TOL[wl.dtype], call


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import medusa_head_speculative_04_b300 as mb
    p = 0x10000  # aligned fake addresses: the call must fail before touching them
    # batch 64 x 5 heads x hidden 16384 in fp32 needs ~21 MB of u alone > the 8 MiB array
    rc = mb.lib.medusa_heads_topk_noalloc(p, p, p, p, None, 64, 16384, 1000, 5, 4, mb.MEDUSA_F32, None, p, p, p,
                                          None)
    assert rc == -6
    assert b"scratch" in mb.lib.medusa_status_string(rc)
