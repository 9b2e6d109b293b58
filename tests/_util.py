"""Shared helpers of the parity tests: comparisons, tolerances, oracle glue."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import synth

# Small bf16 workloads that still span several tiles: ragged kv lengths (including 0),
# a vocabulary that is not a multiple of any tile, GQA, several requests, both head dims.
SMALL_BF16 = synth.Workload("small_bf16", 11, H=512, V=3001, K=3, Hq=8, Hkv=2, D=128, L=0, B=3, dtype="bf16",
                            tree=("cartesian", (3, 2, 2)), ragged=(0, 300))
SMALL_BF16_D64 = dataclasses.replace(SMALL_BF16, name="small_bf16_d64", config_id=12, D=64, Hq=4, Hkv=4,
                                     tree=("seeded", 40, (8, 4, 2)), ragged=(60, 200), B=2, V=2048)
# a query-head group (3) that does not divide 128 takes the mma.sync attention kernel
SMALL_BF16_G3 = dataclasses.replace(SMALL_BF16, name="small_bf16_g3", config_id=13, Hq=6, Hkv=2)

# Float tolerance (max relative error with an rms floor) and near-tie widths.
TOL = {"f32": 1e-4, "bf16": 2e-2}
DELTA = {"f32": 1e-5, "bf16": 1e-3}


def np64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, np.float64)


def npi(t) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def rel_err(g, o) -> float:
    """max_i |g_i - o_i| / max(|o_i|, rms(o))."""
    g, o = np64(g), np64(o)
    if o.size == 0:
        return 0.0
    assert g.shape == o.shape, (g.shape, o.shape)
    if not np.all(np.isfinite(g)):
        return float("inf")
    rms = np.sqrt(np.mean(o * o))
    den = np.maximum(np.abs(o), rms)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(g - o) / den))


def check_topk(ids_g, vals_g, z_o, k, delta):
    """GPU top-k ids must equal the oracle's, except where the oracle's values at the
    two ids differ by less than the near-tie width.  Returns the number of near-ties."""
    ids_g, vals_g = npi(ids_g), np64(vals_g)
    z_o = np64(z_o)
    ids_o, vals_o, _ = oracle.head_topk(z_o, k)
    near = 0
    flat_g, flat_o = ids_g.reshape(-1, k), ids_o.reshape(-1, k)
    zf = z_o.reshape(-1, z_o.shape[-1])
    for r in range(flat_g.shape[0]):
        for t in range(k):
            a, b = flat_g[r, t], flat_o[r, t]
            if a == b:
                continue
            scale = max(1.0, abs(zf[r, b]))
            assert a >= 0 and abs(zf[r, a] - zf[r, b]) < delta * scale, (r, t, a, b, zf[r, a], zf[r, b])
            near += 1
    return near


def step_oracle_inputs(inp):
    """fp64 numpy views of a synth.StepInputs."""
    return {k: np64(getattr(inp, k)) for k in ("h", "W1", "b1", "W2", "lm_head", "X", "q", "k_new", "v_new",
                                               "k_cache", "v_cache") if getattr(inp, k) is not None}


def accept_parity(step, z_o, tokens_g, tt, temperature, thr, alpha, delta, kind, tie_break="first"):
    """Compare the GPU acceptance outputs with the oracle's on the GPU's tree tokens.
    Returns the number of near-tie decisions (outputs may then differ)."""
    acc = oracle.typical_accept(z_o, tokens_g, tt, temperature, thr, alpha, tie_break=tie_break)
    B = tokens_g.shape[0]
    near = 0
    tol = TOL[kind]
    for b in range(B):
        margins = acc["margin"][b][1:]
        if temperature == 0.0:
            tie = np.any(margins < delta * np.maximum(1.0, np.abs(z_o[b]).max()))
        else:
            tie = np.any(margins < delta / temperature)
        tie = tie or acc["joint_margin"][b] < delta
        same = (int(step.accept_len[b]) == acc["accept_len"][b] and int(step.best_node[b]) == acc["best_node"][b]
                and int(step.best_path[b]) == acc["best_path"][b]
                and npi(step.accepted_tokens[b]).tolist() == acc["accepted_tokens"][b].tolist())
        if not same:
            assert tie, (b, int(step.accept_len[b]), acc["accept_len"][b], int(step.best_node[b]), acc["best_node"][b])
            near += 1
            continue
        # next root: greedy token of the winner's logits
        best = acc["best_node"][b]
        zb = z_o[b, best]
        srt = np.sort(zb)
        if int(step.next_root[b]) != acc["next_root"][b]:
            assert srt[-1] - srt[-2] < delta * max(1.0, abs(srt[-1])), b
            near += 1
        if step.node_p is not None:
            p_o = acc["node_p"][b].copy()
            p_o[0] = 1.0
            p_g = np64(step.node_p[b])
            if temperature == 0.0:
                diff = np.nonzero(p_g[1:] != p_o[1:])[0] + 1
                for c in diff:
                    assert acc["margin"][b][c] < delta * max(1.0, abs(z_o[b, tt.parent[c]]).max()), (b, c)
                    near += 1
            else:
                assert rel_err(p_g, p_o) < max(tol, 1e-3), b
    return near
