"""The C ABI library: it loads without a GPU, exports every entry point the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "medusa.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._builder().build()
    import medusa_head_speculative_04_b300 as m
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(medusa_\w+)\s*\(", src)))


def test_header_declares_the_five_step_calls():
    names = declared_functions()
    for n in ("medusa_heads_topk", "medusa_build_tree", "medusa_tree_attention", "medusa_verify_accept",
              "medusa_kv_commit"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib.lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    f = lib.lib.medusa_status_string
    assert f(0) == b"ok"
    assert b"align" in f(-2)
    assert f(-99) == b"unknown status"


def _tree_create(lib, choices):
    flat = [r for c in choices for r in c]
    fa = (ctypes.c_int32 * max(1, len(flat)))(*flat)
    la = (ctypes.c_int32 * max(1, len(choices)))(*[len(c) for c in choices])
    h = ctypes.c_void_p()
    return lib.lib.medusa_tree_create(fa, la, len(choices), ctypes.byref(h))


@pytest.mark.parametrize("bad", [[(0,), (1, 0, 0)], [(0,), (0,)], [(0, -1)], [tuple([0] * 17)]])
def test_tree_create_rejects_bad_specs_on_host(lib, bad):
    # not prefix-closed, duplicate, negative rank, deeper than MEDUSA_MAX_DEPTH
    assert _tree_create(lib, bad) == -1


def test_tree_create_rejects_too_many_nodes(lib):
    choices = [(i,) for i in range(64)] + [(i, j) for i in range(64) for j in range(64)]
    assert _tree_create(lib, choices) == -1


def test_heads_host_validation(lib):
    L = lib.lib
    p = 0x10000  # aligned fake addresses: never dereferenced, the call fails before any launch
    # no workspace: every call below must fail on the host, before any launch
    args = [p] * 5 + [1, 64, 100, 2, 4, 1, None, p, p, p, None, 0, None]
    assert L.medusa_heads_topk(*args) == -4
    bad = list(args)
    bad[0] = None
    assert L.medusa_heads_topk(*bad) == -1
    bad = list(args)
    bad[1] = p + 4
    assert L.medusa_heads_topk(*bad) == -2
    bad = list(args)
    bad[6] = 60          # H not a multiple of 8
    assert L.medusa_heads_topk(*bad) == -3
    bad = list(args)
    bad[9] = 101         # topk > V
    assert L.medusa_heads_topk(*bad) == -1


def test_heads_workspace_size_grows_with_batch(lib):
    f = lib.lib.medusa_heads_topk_workspace_size
    a = f(1, 4096, 32000, 5, 10, 0, 1)
    b = f(16, 4096, 32000, 5, 10, 0, 1)
    assert 0 < a < b
    assert f(0, 4096, 32000, 5, 10, 0, 1) == 0


def test_binding_has_no_cpu_path():
    src = open(os.path.join(ROOT, "medusa_head_speculative_04_b300", "_binding.py")).read()
    assert "import oracle" not in src and "from oracle" not in src
    for f in os.listdir(os.path.join(ROOT, "medusa_head_speculative_04_b300")):
        if f.endswith(".py"):
            s = open(os.path.join(ROOT, "medusa_head_speculative_04_b300", f)).read()
            assert "oracle" not in s.replace("oracle-free", ""), f


def test_heads_workspace_holds_the_tensor_core_buffers(lib):
    """bf16 with three or more batch rows and the root given takes the tensor-core heads
    path, whose workspace also holds the [B,K*H] W1 h buffer and either the top-k
    candidates of every vocabulary tile (k <= 16: tiles 128 to 256 columns wide) or the
    [B,K,V] logits (k > 16); the lm_head-root variant and fp32 stay on the CUDA-core path
    without them."""
    f = lib.lib.medusa_heads_topk_workspace_size
    B, H, V, K, topk = 3, 4096, 32000, 5, 10
    fc = B * K * H * 4
    cand_lo, cand_hi = B * K * (V // 256) * topk * 8, B * K * -(-V // 128) * topk * 8
    tc = f(B, H, V, K, topk, 0, 1)
    assert fc + cand_lo <= tc < fc + cand_hi + B * K * H * 2 + 64 * 1024
    assert tc < B * K * V * 4          # the logits stay out of the workspace
    assert f(B, H, V, K, 17, 0, 1) >= B * K * V * 4 + fc
    base = fc + cand_lo
    assert 0 < f(B, H, V, K, topk, 1, 1) < base
    assert 0 < f(B, H, V, K, topk, 0, 0) < base
    assert 0 < f(2, H, V, K, topk, 0, 1) < base


def test_verify_accept_commit_host_validation(lib):
    """The fused acceptance + commit call rejects missing commit buffers on the host,
    before anything is launched (no tree is needed to get that far)."""
    f = lib.lib.medusa_verify_accept_commit
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf)
    # no k_new: invalid before any launch
    rc = f(None, p, p, p, 1, 4096, 32000, 1, 0.7, 0.09, 0.3, 0, None, None, None, p, p, p, p, p, None,
           None, p, p, p, p, 32, 128, 2112, p, 1 << 20, None)
    assert rc == -1
