"""One Medusa decode step through the five C entry points, with its buffers.

Holds the output and scratch tensors of a fixed workload shape so that a step
allocates nothing and can be captured in a CUDA graph.  The order of the calls
follows the inference flow (wiblog.cn "Medusa multi-head speculative
decoding", section "Inference flow in an online chat service"): heads and
their top-k, candidate tree, tree-masked verification pass, typical
acceptance, commit of the accepted path.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import torch

from . import _binding as mb


class MedusaStep:
    def __init__(self, choices: Sequence[Sequence[int]], B: int, H: int, V: int, K: int, Hq: int, Hkv: int,
                 D: int, Lmax: int, topk: int, dtype: torch.dtype, device="cuda", root_from_lm_head=False,
                 kv_len_hint: int = 0, keep_head_logits=False, keep_logits=False, keep_node_stats=True,
                 rope: bool = False, rope_theta: float = 10000.0, tie_break: str = "first"):
        self.tree = mb.Tree(choices)
        self.B, self.H, self.V, self.K = B, H, V, K
        self.Hq, self.Hkv, self.D, self.Lmax, self.topk = Hq, Hkv, D, Lmax, topk
        self.dtype, self.device = dtype, torch.device(device)
        self.root_from_lm_head = root_from_lm_head
        self.kv_len_hint = kv_len_hint
        # rope: the tree's q and k are rotated at the position ids the tree expansion
        # produced, and the rotated keys are what the commit appends to the cache
        self.rope, self.rope_theta = rope, rope_theta
        self.tie_break = tie_break  # among equally deep accepted nodes: "first" in order or "joint" probability
        T, P, W = self.tree.T, self.tree.P, self.tree.dmax + 1
        dc = mb.MEDUSA_BF16 if dtype == torch.bfloat16 else mb.MEDUSA_F32
        i32 = dict(dtype=torch.int32, device=self.device)
        f32 = dict(dtype=torch.float32, device=self.device)
        self.topk_ids = torch.zeros(B, K, topk, **i32)
        self.topk_vals = torch.zeros(B, K, topk, **f32)
        self.root = torch.zeros(B, **i32)
        self.tokens = torch.zeros(B, T, **i32)
        self.positions = torch.zeros(B, T, **i32)
        self.candidates = torch.zeros(B, P, W, **i32)
        self.attn_out = torch.zeros(B, T, Hq, D, **f32)
        self.k_rot = torch.zeros(B, T, Hkv, D, dtype=dtype, device=self.device) if rope else None
        # the per-request results share one buffer, so a caller can read them with one copy;
        # each part starts on a 16-byte boundary, as the C entry points require
        Bp = (B + 3) // 4 * 4
        self.results = torch.zeros(4 * Bp + B * W, **i32)
        self.accept_len = self.results[0:B]
        self.best_path = self.results[Bp:Bp + B]
        self.best_node = self.results[2 * Bp:2 * Bp + B]
        self.next_root = self.results[3 * Bp:3 * Bp + B]
        self.accepted_tokens = self.results[4 * Bp:].view(B, W)
        self.dev_status = torch.zeros(B, **i32)
        self.head_logits = torch.zeros(B, K, V, **f32) if keep_head_logits else None
        self.logits = torch.zeros(B, T, V, **f32) if keep_logits else None
        self.node_p = torch.zeros(B, T, **f32) if keep_node_stats else None
        self.node_H = torch.zeros(B, T, **f32) if keep_node_stats else None
        self.ws_heads = mb.workspace(mb.medusa_heads_topk_workspace_size(B, H, V, K, topk, root_from_lm_head, dc),
                                     self.device)
        self.ws_attn = mb.workspace(mb.medusa_tree_attention_workspace_size(self.tree, B, Hq, Hkv, D, Lmax,
                                                                            kv_len_hint, dc), self.device)
        self.ws_verify = mb.workspace(mb.medusa_verify_accept_workspace_size(self.tree, B, H, V, dc), self.device)
        self.ws_tree_heads = None  # allocated on the first heads_from_tree call

    @property
    def T(self) -> int:
        return self.tree.T

    def heads(self, h, W1, b1, W2, lm_head=None, stream=None):
        mb.medusa_heads_topk(h, W1, b1, W2, lm_head if self.root_from_lm_head else None, self.topk,
                             self.topk_ids, self.topk_vals, self.root, self.ws_heads,
                             head_logits=self.head_logits, stream=stream)

    def heads_from_tree(self, X, W1, b1, W2, stream=None):
        """Next step's candidates from the heads on the tree nodes' states X (the
        verification input): the top-k of each request's accepted node go to
        ``topk_ids``/``topk_vals`` and its next token to ``root``, so the next
        :meth:`build` continues from the accepted branch."""
        if self.ws_tree_heads is None:
            dc = mb.MEDUSA_BF16 if self.dtype == torch.bfloat16 else mb.MEDUSA_F32
            self.ws_tree_heads = mb.workspace(mb.medusa_heads_topk_tree_workspace_size(
                self.tree, self.B, self.H, self.V, self.K, self.topk, dc), self.device)
        mb.medusa_heads_topk_tree(self.tree, X, W1, b1, W2, self.best_node, self.topk, self.topk_ids,
                                  self.topk_vals, self.ws_tree_heads, head_logits=self.head_logits, stream=stream)
        self.root.copy_(self.next_root)

    def build(self, kv_len, root=None, stream=None):
        mb.medusa_build_tree(self.tree, self.root if root is None else root, self.topk_ids, kv_len, self.tokens,
                             self.positions, self.candidates, self.dev_status, stream=stream)

    def attention(self, q, k_new, v_new, k_cache, v_cache, kv_len, stream=None):
        mb.medusa_tree_attention(self.tree, q, k_new, v_new, k_cache, v_cache, kv_len, self.attn_out,
                                 self.ws_attn, 1.0 / math.sqrt(self.D), kv_len_hint=self.kv_len_hint,
                                 dev_status=self.dev_status, stream=stream, position_ids=self.positions,
                                 rope=self.rope, rope_theta=self.rope_theta, k_rot=self.k_rot)

    def verify(self, X, lm_head, temperature: float, threshold: float = 0.09, alpha: float = 0.3, stream=None):
        mb.medusa_verify_accept(self.tree, X, lm_head, self.tokens, temperature, threshold, alpha,
                                self.accept_len, self.best_path, self.best_node, self.accepted_tokens,
                                self.next_root, self.ws_verify, logits=self.logits, node_p=self.node_p,
                                node_H=self.node_H, dev_status=self.dev_status, stream=stream,
                                tie_break=self.tie_break)

    def verify_commit(self, X, lm_head, k_new, v_new, k_cache, v_cache, kv_len, temperature: float,
                      threshold: float = 0.09, alpha: float = 0.3, stream=None):
        """:meth:`verify` and :meth:`commit` with one launch fewer (the acceptance's CTA
        of a request also commits its accepted rows)."""
        mb.medusa_verify_accept_commit(self.tree, X, lm_head, self.tokens, temperature, threshold, alpha,
                                       self.accept_len, self.best_path, self.best_node, self.accepted_tokens,
                                       self.next_root, self.k_rot if self.rope else k_new, v_new, k_cache, v_cache,
                                       kv_len, self.ws_verify, logits=self.logits, node_p=self.node_p,
                                       node_H=self.node_H, dev_status=self.dev_status, stream=stream,
                                       tie_break=self.tie_break)

    def commit(self, k_new, v_new, k_cache, v_cache, kv_len, stream=None):
        mb.medusa_kv_commit(self.tree, self.k_rot if self.rope else k_new, v_new, k_cache, v_cache, kv_len,
                            self.best_node,
                            dev_status=self.dev_status, stream=stream)

    def run(self, h, W1, b1, W2, lm_head, X, q, k_new, v_new, k_cache, v_cache, kv_len, temperature: float,
            threshold: float = 0.09, alpha: float = 0.3, root: Optional[torch.Tensor] = None, stream=None):
        """One whole step.  ``root`` (int32 [B], device) is the previous step's next token; it is
        copied into ``self.root`` and ignored when the step derives the root from lm_head(h)."""
        if root is not None and not self.root_from_lm_head:
            self.root.copy_(root)
        self.heads(h, W1, b1, W2, lm_head, stream=stream)
        self.build(kv_len, stream=stream)
        self.attention(q, k_new, v_new, k_cache, v_cache, kv_len, stream=stream)
        self.verify_commit(X, lm_head, k_new, v_new, k_cache, v_cache, kv_len, temperature, threshold, alpha,
                           stream=stream)

    def capture(self, *args, prologue=None, epilogue=None, stream: Optional[torch.cuda.Stream] = None, **kwargs):
        """Capture one whole step (the arguments of :meth:`run`) in a CUDA graph.

        The graph reads the tensors it was captured with: refill them in place and
        ``replay()`` it to run the next step with one launch from the host.
        ``prologue`` and ``epilogue`` (callables, or None) are captured just before
        and just after the step, on the same stream.  The returned graph holds
        references to the arguments and to both callables (and so to the tensors
        their closures use), so no buffer it reads can be freed and reused while it
        lives.  One eager step runs first, so its outputs change state (``kv_len``
        and the cache rows it commits) like any other step.
        """
        cur = torch.cuda.current_stream(self.device)
        s = stream if stream is not None else torch.cuda.Stream(self.device)  # capture needs a side stream
        s.wait_stream(cur)
        with torch.cuda.stream(s):
            if prologue is not None:
                prologue()
            self.run(*args, **kwargs)     # sets the kernels' attributes outside the capture
            if epilogue is not None:
                epilogue()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            if prologue is not None:
                prologue()
            self.run(*args, **kwargs)
            if epilogue is not None:
                epilogue()
        cur.wait_stream(s)
        g.medusa_keepalive = (args, kwargs, prologue, epilogue)
        return g
