"""ctypes binding of the C ABI declared in include/medusa.h.

Argument marshalling only: every step of the decode step runs in the CUDA
kernels of libmedusa_b300.so.  Each function has the C entry point's name and
takes torch tensors (device memory owned by PyTorch) plus the scalars of the C
call; it raises MedusaError when the library reports a host-side error.
There is no CPU path: if the shared library is missing, importing this module
fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmedusa_b300.so")

MEDUSA_F32 = 0
MEDUSA_BF16 = 1
DEV_KV_OVERFLOW = 1
DEV_NAN = 2
DEV_TIMEOUT = 4
DEV_BAD_TOKEN = 8
MAX_DEPTH = 16


class MedusaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({lib.medusa_status_string(code).decode()})")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build the CUDA library first "
            "(python medusa_head_speculative_04_b300/build.py)")
    return ctypes.CDLL(_LIB_PATH)


lib = _load()

_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t


class TreeInfo(ctypes.Structure):
    _fields_ = [("T", _i32), ("P", _i32), ("dmax", _i32), ("mask_words", _i32),
                ("max_rank", _i32 * MAX_DEPTH)]


def _sig(name, restype, argtypes):
    f = getattr(lib, name)
    f.restype = restype
    f.argtypes = argtypes
    return f


_sig("medusa_status_string", ctypes.c_char_p, [ctypes.c_int])
_sig("medusa_kernel_launches", ctypes.c_uint64, [])
_sig("medusa_tree_create", ctypes.c_int, [_vp, _vp, _i32, ctypes.POINTER(_vp)])
_sig("medusa_tree_get_info", ctypes.c_int, [_vp, ctypes.POINTER(TreeInfo)])
_sig("medusa_tree_copy_tables", ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp])
_sig("medusa_tree_destroy", None, [_vp])
_sig("medusa_heads_topk_workspace_size", _sz, [_i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int])
_sig("medusa_heads_topk", ctypes.c_int,
     [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _sz, _vp])
_sig("medusa_heads_topk_noalloc", ctypes.c_int,
     [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _vp, _vp, _vp, _vp, _vp])
_sig("medusa_heads_topk_tree_workspace_size", _sz, [_vp, _i32, _i32, _i32, _i32, _i32, ctypes.c_int])
_sig("medusa_heads_topk_tree", ctypes.c_int,
     [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _vp, _vp, _vp, _vp, _sz, _vp])
_sig("medusa_build_tree", ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp])
_sig("medusa_tree_attention_workspace_size", _sz, [_vp, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int])
_sig("medusa_tree_attention", ctypes.c_int,
     [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _f32, ctypes.c_int, _vp,
      _vp, _vp, _sz, _vp, _vp])
_sig("medusa_tree_query", ctypes.c_int, [_vp, _vp, _vp, _vp, _vp])
_sig("medusa_verify_accept_workspace_size", _sz, [_vp, _i32, _i32, _i32, ctypes.c_int])
_sig("medusa_verify_accept", ctypes.c_int,
     [_vp, _vp, _vp, _vp, _i32, _i32, _i32, ctypes.c_int, _f32, _f32, _f32, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
      _vp, _vp, _vp, _vp, _sz, _vp])
_sig("medusa_sample_next", ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _f32, _f32, _vp, _vp])
_sig("medusa_verify_accept_commit", ctypes.c_int,
     [_vp, _vp, _vp, _vp, _i32, _i32, _i32, ctypes.c_int, _f32, _f32, _f32, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
      _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _sz, _vp])
_sig("medusa_kv_commit", ctypes.c_int,
     [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_int, _vp, _vp])


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise MedusaError(fn, rc)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the Medusa library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MEDUSA_F32
    if t.dtype == torch.bfloat16:
        return MEDUSA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


class Tree:
    """A fixed candidate tree (medusa_tree_create); tables live on the current device."""

    def __init__(self, choices: Sequence[Sequence[int]]):
        flat = [int(r) for c in choices for r in c]
        lens = [len(c) for c in choices]
        fa = (_i32 * max(1, len(flat)))(*flat)
        la = (_i32 * max(1, len(lens)))(*lens)
        h = _vp()
        _check("medusa_tree_create", lib.medusa_tree_create(fa, la, len(lens), ctypes.byref(h)))
        self._h = h
        info = TreeInfo()
        _check("medusa_tree_get_info", lib.medusa_tree_get_info(h, ctypes.byref(info)))
        self.T, self.P, self.dmax, self.mask_words = info.T, info.P, info.dmax, info.mask_words
        self.max_rank = list(info.max_rank)[: self.dmax]

    @property
    def handle(self):
        return self._h

    def query(self):
        """(T, P, dmax, top-k each head must supply) from medusa_tree_query."""
        T, P, dm = _i32(), _i32(), _i32()
        tk = (_i32 * MAX_DEPTH)()
        _check("medusa_tree_query", lib.medusa_tree_query(self._h, ctypes.byref(T), ctypes.byref(P), ctypes.byref(dm), tk))
        return T.value, P.value, dm.value, list(tk)[: dm.value]

    def tables(self):
        T, P, W, MW = self.T, self.P, self.dmax + 1, self.mask_words
        parent, depth, rank = (_i32 * T)(), (_i32 * T)(), (_i32 * T)()
        mask = (ctypes.c_uint32 * (T * MW))()
        paths = (_i32 * (P * W))()
        _check("medusa_tree_copy_tables", lib.medusa_tree_copy_tables(self._h, parent, depth, rank, mask, paths))
        return dict(parent=list(parent), depth=list(depth), rank=list(rank),
                    mask=[list(mask[i * MW:(i + 1) * MW]) for i in range(T)],
                    paths=[list(paths[p * W:(p + 1) * W]) for p in range(P)])

    def close(self):
        if getattr(self, "_h", None):
            lib.medusa_tree_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kernel_launches() -> int:
    """Kernels launched (or captured) by the library in this process so far."""
    return int(lib.medusa_kernel_launches())


def workspace(nbytes: int, device) -> torch.Tensor:
    """Zero-filled scratch buffer for one entry point (16-byte aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def medusa_heads_topk_workspace_size(B, H, V, K, topk, with_lm_head, dtype_c) -> int:
    return lib.medusa_heads_topk_workspace_size(B, H, V, K, topk, int(bool(with_lm_head)), dtype_c)


def medusa_heads_topk(h, w1, b1, w2, lm_head, topk: int, topk_ids, topk_vals, root_tok, ws,
                      head_logits=None, stream=None) -> None:
    B, H = h.shape
    K, V = w2.shape[0], w2.shape[1]
    _check("medusa_heads_topk", lib.medusa_heads_topk(
        _ptr(h), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(lm_head), B, H, V, K, topk, dtype_code(h),
        _ptr(head_logits), _ptr(topk_ids), _ptr(topk_vals), _ptr(root_tok), _ptr(ws), ws.numel(),
        _stream(stream)))


def medusa_heads_topk_noalloc(h, w1, b1, w2, lm_head, topk: int, topk_ids, topk_vals, root_tok,
                              head_logits=None, stream=None) -> None:
    """medusa_heads_topk without a workspace, for callers that cannot allocate device memory
    (the scratch is a fixed array inside the library, shared by every call)."""
    B, H = h.shape
    K, V = w2.shape[0], w2.shape[1]
    _check("medusa_heads_topk_noalloc", lib.medusa_heads_topk_noalloc(
        _ptr(h), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(lm_head), B, H, V, K, topk, dtype_code(h),
        _ptr(head_logits), _ptr(topk_ids), _ptr(topk_vals), _ptr(root_tok), _stream(stream)))


def medusa_heads_topk_tree_workspace_size(tree: Tree, B, H, V, K, topk, dtype_c) -> int:
    return lib.medusa_heads_topk_tree_workspace_size(tree.handle, B, H, V, K, topk, dtype_c)


def medusa_heads_topk_tree(tree: Tree, x, w1, b1, w2, best_node, topk: int, topk_ids, topk_vals, ws,
                           head_logits=None, stream=None) -> None:
    B, T, H = x.shape
    K, V = w2.shape[0], w2.shape[1]
    _check("medusa_heads_topk_tree", lib.medusa_heads_topk_tree(
        tree.handle, _ptr(x), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(best_node), B, H, V, K, topk, dtype_code(x),
        _ptr(head_logits), _ptr(topk_ids), _ptr(topk_vals), _ptr(ws), ws.numel(), _stream(stream)))


def medusa_build_tree(tree: Tree, root_tok, topk_ids, kv_len, tree_tokens, position_ids,
                      candidates=None, dev_status=None, stream=None) -> None:
    B, K, topk = topk_ids.shape
    _check("medusa_build_tree", lib.medusa_build_tree(
        tree.handle, _ptr(root_tok), _ptr(topk_ids), B, K, topk, _ptr(kv_len), _ptr(tree_tokens),
        _ptr(position_ids), _ptr(candidates), _ptr(dev_status), _stream(stream)))


def medusa_tree_attention_workspace_size(tree: Tree, B, Hq, Hkv, D, Lmax, kv_len_hint, dtype_c) -> int:
    return lib.medusa_tree_attention_workspace_size(tree.handle, B, Hq, Hkv, D, Lmax, kv_len_hint, dtype_c)


def medusa_tree_attention(tree: Tree, q, k_new, v_new, k_cache, v_cache, kv_len, out, ws, scale: float,
                          kv_len_hint: int = 0, dev_status=None, stream=None, position_ids=None, rope: bool = False,
                          rope_theta: float = 10000.0, k_rot=None) -> None:
    B, T, Hq, D = q.shape
    Hkv = k_new.shape[2]
    Lmax = k_cache.shape[2]
    _check("medusa_tree_attention", lib.medusa_tree_attention(
        tree.handle, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len),
        _ptr(position_ids), B, Hq, Hkv, D, Lmax, kv_len_hint, scale, int(bool(rope)), rope_theta, dtype_code(q),
        _ptr(out), _ptr(k_rot), _ptr(ws), ws.numel() if ws is not None else 0, _ptr(dev_status), _stream(stream)))


def medusa_verify_accept_workspace_size(tree: Tree, B, H, V, dtype_c) -> int:
    return lib.medusa_verify_accept_workspace_size(tree.handle, B, H, V, dtype_c)


def medusa_verify_accept(tree: Tree, x, lm_head, tree_tokens, temperature: float, posterior_threshold: float,
                         posterior_alpha: float, accept_len, best_path, best_node, accepted_tokens, next_root,
                         ws, logits=None, node_p=None, node_H=None, dev_status=None, stream=None,
                         tie_break: str = "first") -> None:
    B, T, H = x.shape
    V = lm_head.shape[0]
    tb = {"first": 0, "joint": 1}[tie_break]
    _check("medusa_verify_accept", lib.medusa_verify_accept(
        tree.handle, _ptr(x), _ptr(lm_head), _ptr(tree_tokens), B, H, V, dtype_code(x), temperature,
        posterior_threshold, posterior_alpha, tb, _ptr(logits), _ptr(node_p), _ptr(node_H), _ptr(accept_len),
        _ptr(best_path), _ptr(best_node), _ptr(accepted_tokens), _ptr(next_root), _ptr(dev_status), _ptr(ws),
        ws.numel(), _stream(stream)))


def medusa_verify_accept_commit(tree: Tree, x, lm_head, tree_tokens, temperature: float, posterior_threshold: float,
                                posterior_alpha: float, accept_len, best_path, best_node, accepted_tokens, next_root,
                                k_new, v_new, k_cache, v_cache, kv_len, ws, logits=None, node_p=None, node_H=None,
                                dev_status=None, stream=None, tie_break: str = "first") -> None:
    """medusa_verify_accept and the KV commit of its winner in one launch sequence."""
    B, T, H = x.shape
    V = lm_head.shape[0]
    _, Hkv, Lmax, D = k_cache.shape
    tb = {"first": 0, "joint": 1}[tie_break]
    _check("medusa_verify_accept_commit", lib.medusa_verify_accept_commit(
        tree.handle, _ptr(x), _ptr(lm_head), _ptr(tree_tokens), B, H, V, dtype_code(x), temperature,
        posterior_threshold, posterior_alpha, tb, _ptr(logits), _ptr(node_p), _ptr(node_H), _ptr(accept_len),
        _ptr(best_path), _ptr(best_node), _ptr(accepted_tokens), _ptr(next_root), _ptr(dev_status), _ptr(k_new),
        _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), Hkv, D, Lmax, _ptr(ws), ws.numel(),
        _stream(stream)))


def medusa_kv_commit(tree: Tree, k_new, v_new, k_cache, v_cache, kv_len, best_node, dev_status=None,
                     stream=None) -> None:
    B, Hkv, Lmax, D = k_cache.shape
    _check("medusa_kv_commit", lib.medusa_kv_commit(
        tree.handle, _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(best_node), B,
        Hkv, D, Lmax, dtype_code(k_cache), _ptr(dev_status), _stream(stream)))


def medusa_sample_next(tree: Tree, logits, best_node, uniform, temperature: float, top_p: float, next_token,
                       stream=None) -> None:
    B, T, V = logits.shape
    _check("medusa_sample_next", lib.medusa_sample_next(
        tree.handle, _ptr(logits), _ptr(best_node), _ptr(uniform), B, V, temperature, top_p, _ptr(next_token),
        _stream(stream)))
