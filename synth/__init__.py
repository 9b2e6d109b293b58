"""Seeded synthetic inputs for the Medusa decode step.

Both the CUDA path and the CPU oracle draw their inputs from this module, and
nothing else is shared between them.  It holds none of the step's arithmetic:
only a counter-based generator, input rounding to bf16, the seeded tree-choice
generators, the workload table and the assembly of one step's inputs.

Generator.  Element ``e`` of a tensor keyed by ``seed`` is built from three
splitmix64 outputs (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): output ``c`` is ``mix(seed + (c + 1) * golden)``,
taken at counters ``3e, 3e+1, 3e+2``.  Their twelve 16-bit fields are summed
(the classic "sum of twelve uniforms" approximation of a standard normal) and
centred and scaled by powers of two, so the value is an exact small integer
times 2**-16 before one float32 multiply by the standard deviation.  Integer
ops and a single IEEE multiply give bit-identical tensors on the CPU and on a
GPU, and any element can be regenerated alone from its flat index.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional, Sequence, Tuple

import torch

_GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB
_U64 = (1 << 64) - 1
SEED_BASE = 0x4D45445553410000          # "MEDUSA\0\0"
_SUM12_MEAN = 12 * 65535 // 2           # 393210: mean of twelve 16-bit fields
_CHUNK = 1 << 24


def _s64(c: int) -> int:
    """Unsigned 64-bit constant as the int64 with the same bits."""
    c &= _U64
    return c - (1 << 64) if c >= (1 << 63) else c


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(_MIX1)
    z = (z ^ _srl(z, 27)) * _s64(_MIX2)
    return z ^ _srl(z, 31)


def splitmix64_py(seed: int, counter: int) -> int:
    """Output number ``counter`` (0-based) of splitmix64 started at ``seed``."""
    z = (seed + (counter + 1) * _GOLDEN) & _U64
    z = ((z ^ (z >> 30)) * _MIX1) & _U64
    z = ((z ^ (z >> 27)) * _MIX2) & _U64
    return z ^ (z >> 31)


class SplitMix64:
    """Sequential splitmix64 stream for small integer draws (trees, lengths)."""

    def __init__(self, seed: int):
        self.seed = seed & _U64
        self.n = 0

    def next(self) -> int:
        v = splitmix64_py(self.seed, self.n)
        self.n += 1
        return v

    def below(self, n: int) -> int:
        return self.next() % n


def tensor_seed(config_id: int, tensor_id: int) -> int:
    return (SEED_BASE ^ (config_id << 32) ^ (tensor_id << 16)) & _U64


def normal_at(seed: int, flat_index: torch.Tensor, std: float) -> torch.Tensor:
    """Approximate N(0, std^2) float32 values at the given flat element indices."""
    idx = flat_index.to(torch.int64)
    base = _s64(seed)
    s = torch.zeros_like(idx)
    for j in range(3):
        ctr = idx * 3 + (j + 1)
        z = _mix(base + ctr * _s64(_GOLDEN))
        s = s + (z & 0xFFFF) + ((z >> 16) & 0xFFFF) + ((z >> 32) & 0xFFFF) + _srl(z, 48)
    x = (s - _SUM12_MEAN).to(torch.float32) * (1.0 / 65536.0)
    return x * torch.tensor(std, dtype=torch.float32, device=x.device)


def normal(shape: Sequence[int], seed: int, std: float = 1.0,
           dtype: torch.dtype = torch.float32, device="cpu") -> torch.Tensor:
    """Tensor of the generator's values, rounded to ``dtype`` (RNE)."""
    n = 1
    for d in shape:
        n *= int(d)
    out = torch.empty(n, dtype=dtype, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        idx = torch.arange(s, e, dtype=torch.int64, device=device)
        out[s:e] = normal_at(seed, idx, std).to(dtype)
    return out.view(*shape)


def round_bf16(x: torch.Tensor) -> torch.Tensor:
    """float32 tensor holding the bf16-rounded (RNE) values of ``x``."""
    return x.to(torch.bfloat16).to(torch.float32)


# --------------------------------------------------------------------------
# Trees ("medusa_choices": one tuple of per-depth ranks per candidate node)
# --------------------------------------------------------------------------

def cartesian_choices(ks: Sequence[int]) -> List[Tuple[int, ...]]:
    """Every rank tuple of the full product tree top-ks[0] x top-ks[1] x ..."""
    out: List[Tuple[int, ...]] = []
    level: List[Tuple[int, ...]] = [()]
    for k in ks:
        level = [p + (r,) for p in level for r in range(k)]
        out.extend(level)
    return out


def seeded_sparse_choices(n_nodes: int, fanout: Sequence[int], seed: int) -> List[Tuple[int, ...]]:
    """Seeded sparse tree: all root children, then uniform picks from the frontier.

    ``fanout[d]`` bounds the number of children of a node at depth ``d`` (the
    root is depth 0) and ``len(fanout)`` bounds the depth.  Children are added
    in rank order, so every node's child ranks are 0..c-1.
    """
    rng = SplitMix64(seed)
    nodes: List[Tuple[int, ...]] = [(r,) for r in range(min(fanout[0], n_nodes))]
    nchild: Dict[Tuple[int, ...], int] = {(): len(nodes)}
    for n in nodes:
        nchild[n] = 0

    def frontier() -> List[Tuple[int, ...]]:
        f = []
        for n in nodes:
            d = len(n)
            if d < len(fanout) and nchild[n] < fanout[d]:
                f.append(n + (nchild[n],))
        f.sort(key=lambda t: (len(t), t))
        return f

    while len(nodes) < n_nodes:
        f = frontier()
        if not f:
            break
        pick = f[rng.below(len(f))]
        nodes.append(pick)
        nchild[pick] = 0
        nchild[pick[:-1]] += 1
    return nodes


def canonical_order(choices: Sequence[Tuple[int, ...]]) -> List[Tuple[int, ...]]:
    """Node layout used for every per-node tensor: root first, then by depth, then by rank tuple."""
    return [()] + sorted((tuple(c) for c in choices), key=lambda t: (len(t), t))


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    H: int
    V: int
    K: int
    Hq: int
    Hkv: int
    D: int
    L: int
    B: int
    dtype: str                      # "f32" or "bf16"
    tree: Tuple                     # ("cartesian", ks) or ("seeded", n, fanout)
    temperatures: Tuple[float, ...] = (0.0, 0.7)
    ragged: Optional[Tuple[int, int]] = None   # kv lengths uniform in [lo, hi]
    lmax_slack: int = 64
    w_std: float = 0.02
    posterior_threshold: float = 0.09
    posterior_alpha: float = 0.3
    topk: int = 0                   # per-head top-k kept; 0 = largest rank in the tree + 1

    @property
    def Lmax(self) -> int:
        hi = self.ragged[1] if self.ragged else self.L
        return hi + self.lmax_slack

    def choices(self) -> List[Tuple[int, ...]]:
        if self.tree[0] == "cartesian":
            return cartesian_choices(self.tree[1])
        _, n, fan = self.tree
        fan = tuple(fan)[: self.K]
        return seeded_sparse_choices(n, fan, tensor_seed(self.config_id, 0x7E))

    def k_needed(self) -> int:
        if self.topk:
            return self.topk
        return 1 + max((r for c in self.choices() for r in c), default=0)

    def kv_lens(self) -> List[int]:
        if not self.ragged:
            return [self.L] * self.B
        lo, hi = self.ragged
        rng = SplitMix64(tensor_seed(self.config_id, 0x4C))
        return [lo + rng.below(hi - lo + 1) for _ in range(self.B)]


TREE64 = ("seeded", 64, (10, 6, 4, 2, 1))

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, H=256, V=1000, K=3, Hq=4, Hkv=4, D=64, L=128, B=1,
                     dtype="f32", tree=("cartesian", (2, 3)), lmax_slack=8),
    "vicuna7b": Workload("vicuna7b", 2, H=4096, V=32000, K=5, Hq=32, Hkv=32, D=128,
                         L=2048, B=1, dtype="bf16", tree=TREE64),
    "llama8b_b1": Workload("llama8b_b1", 3, H=4096, V=128256, K=5, Hq=32, Hkv=8, D=128,
                           L=8192, B=1, dtype="bf16", tree=TREE64),
    "llama8b_b4": Workload("llama8b_b4", 3, H=4096, V=128256, K=5, Hq=32, Hkv=8, D=128,
                           L=8192, B=4, dtype="bf16", tree=TREE64),
    "llama8b_b16": Workload("llama8b_b16", 3, H=4096, V=128256, K=5, Hq=32, Hkv=8, D=128,
                            L=8192, B=16, dtype="bf16", tree=TREE64),
    "ragged7b": Workload("ragged7b", 4, H=4096, V=32000, K=4, Hq=32, Hkv=32, D=128,
                         L=0, B=16, dtype="bf16", tree=TREE64, temperatures=(0.7,),
                         ragged=(512, 8192)),
    "wide70b": Workload("wide70b", 5, H=8192, V=128256, K=3, Hq=64, Hkv=8, D=128,
                        L=4096, B=1, dtype="bf16", tree=("cartesian", (10, 10, 10))),
}


# tensor ids inside one workload's seed space
TID = dict(h=1, W1=2, b1=3, W2=4, lm_head=5, X=6, q=7, k_new=8, v_new=9,
           k_cache=10, v_cache=11, root=12, plant_tok=13, plant_depth=14, X_noise=15)


@dataclass
class StepInputs:
    """One step's inputs.  Float tensors hold values already rounded to ``dtype``."""
    wl: Workload
    choices: List[Tuple[int, ...]]
    dtype: torch.dtype
    h: torch.Tensor
    W1: torch.Tensor
    b1: torch.Tensor
    W2: torch.Tensor
    lm_head: torch.Tensor
    X: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    kv_len: torch.Tensor            # int32 [B]
    root: torch.Tensor              # int32 [B]
    plant: Optional[Dict] = None
    extra: Dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return len(self.choices) + 1

    def to(self, device) -> "StepInputs":
        """The same inputs with every tensor copied to ``device`` (values unchanged)."""
        moved = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in self.__dict__.items()}
        return StepInputs(**moved)


def torch_dtype(wl: Workload) -> torch.dtype:
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def make_inputs(wl: Workload, device="cpu", variant: str = "random",
                plant_depth: Optional[int] = None, with_weights: bool = True) -> StepInputs:
    """Assemble one step's seeded inputs on ``device``.

    variant:
      "random"  every tensor from the generator;
      "zeroinit" W1 = b1 = 0 and every W2_k a copy of lm_head (the heads' start state);
      "plant"   request b's heads are given a clear top-1 token per depth (a W2 row
                along h_b) and the tree-node states on the rank-0 chain are steered
                toward the next planted token, so acceptance runs several levels deep.
    """
    dt = torch_dtype(wl)
    cid = wl.config_id
    choices = wl.choices()
    T = len(choices) + 1
    B, H, V, K = wl.B, wl.H, wl.V, wl.K
    g = lambda name, shape, std: normal(shape, tensor_seed(cid, TID[name]), std, dt, device)

    h = g("h", (B, H), 1.0)
    if with_weights:
        W1 = g("W1", (K, H, H), wl.w_std)
        b1 = g("b1", (K, H), wl.w_std)
        W2 = g("W2", (K, V, H), wl.w_std)
        lm_head = g("lm_head", (V, H), wl.w_std)
    else:
        W1 = b1 = W2 = lm_head = None
    X = g("X", (B, T, H), 1.0)
    q = g("q", (B, T, wl.Hq, wl.D), 1.0)
    k_new = g("k_new", (B, T, wl.Hkv, wl.D), 1.0)
    v_new = g("v_new", (B, T, wl.Hkv, wl.D), 1.0)
    k_cache = g("k_cache", (B, wl.Hkv, wl.Lmax, wl.D), 1.0)
    v_cache = g("v_cache", (B, wl.Hkv, wl.Lmax, wl.D), 1.0)
    kv_len = torch.tensor(wl.kv_lens(), dtype=torch.int32, device=device)
    rr = SplitMix64(tensor_seed(cid, TID["root"]))
    root = torch.tensor([rr.below(V) for _ in range(B)], dtype=torch.int32, device=device)

    inp = StepInputs(wl, choices, dt, h, W1, b1, W2, lm_head, X, q, k_new, v_new,
                     k_cache, v_cache, kv_len, root)
    if variant == "zeroinit":
        assert with_weights
        inp.W1 = torch.zeros_like(W1)
        inp.b1 = torch.zeros_like(b1)
        inp.W2 = lm_head.unsqueeze(0).expand(K, V, H).contiguous()
    elif variant == "plant":
        assert with_weights
        _plant(inp, plant_depth)
    elif variant != "random":
        raise ValueError(variant)
    return inp


def _plant(inp: StepInputs, plant_depth: Optional[int]) -> None:
    wl = inp.wl
    order = canonical_order(inp.choices)
    index = {c: i for i, c in enumerate(order)}
    chain = []                                   # canonical indices of (), (0,), (0,0), ...
    t = ()
    while t in index:
        chain.append(index[t])
        t = t + (0,)
    max_d = len(chain) - 1                       # deepest rank-0 node
    K, V, H, B = wl.K, wl.V, wl.H, wl.B
    rt = SplitMix64(tensor_seed(wl.config_id, TID["plant_tok"]))
    rd = SplitMix64(tensor_seed(wl.config_id, TID["plant_depth"]))
    dev = inp.h.device
    W2 = inp.W2.clone()
    X = inp.X.clone()
    lm32 = inp.lm_head.to(torch.float32)
    depths, toks = [], []
    used = set()
    for b in range(B):
        d_b = plant_depth if plant_depth is not None else rd.below(max_d + 1)
        d_b = min(d_b, max_d, K)
        tk = []
        for d in range(1, d_b + 1):
            while True:
                v = rt.below(V)
                if (d, v) not in used:
                    break
            used.add((d, v))
            tk.append(v)
        hb = inp.h[b].to(torch.float32)
        hunit = hb / hb.norm()
        for d, v in enumerate(tk, start=1):
            W2[d - 1, v] = (0.5 * hunit).to(inp.dtype)
        for d, v in enumerate(tk):               # node at depth d steers toward depth d+1's token
            w = lm32[v]
            noise = normal((H,), tensor_seed(wl.config_id, TID["X_noise"]) ^ (b << 8) ^ d, 0.1,
                           torch.float32, dev)
            X[b, chain[d]] = (8.0 * w / w.norm() + noise).to(inp.dtype)
        depths.append(d_b)
        toks.append(tk)
    inp.W2 = W2
    inp.X = X
    inp.plant = dict(depths=depths, tokens=toks, chain=chain)
