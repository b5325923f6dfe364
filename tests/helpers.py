"""Shared test utilities: workloads on the device, oracle references and the
comparison rules.

Comparison rules (the selection tolerance is the one the method's acceptance
criteria fix; the attention bounds likewise):
  R1  top-k lists and unions are bit-exact when both sides select from the
      same fp32 score matrix;
  R2  end to end, a selected block may differ from the fp64 oracle's only
      where its fp64 score lies within 1e-4 * max(1, |s_K|) of the k-th
      fp64 score s_K (absolute below 1, relative above);
  R3  attention on identical block lists: max |O - O64| <= 2e-2 and
      mean |O - O64| <= 2e-3, |lse - lse64| <= 1e-3.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth

R2_TOL = 1e-4
R3_MAX, R3_MEAN, R3_LSE = 2e-2, 2e-3, 1e-3


def to_dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def dev_inputs(inp: dict, device="cuda") -> dict:
    wl = inp["workload"]
    d = {"Q": to_dev(inp["Q"], device)}
    if wl.page_size:
        pt = inp["page_table"]
        d["K"] = to_dev(synth.to_paged(inp["K"], pt, wl.page_size), device)
        d["V"] = to_dev(synth.to_paged(inp["V"], pt, wl.page_size), device)
        d["page_table"] = torch.from_numpy(pt).to(device)
    else:
        d["K"] = to_dev(inp["K"], device)
        d["V"] = to_dev(inp["V"], device)
        d["page_table"] = None
    return d


def widened(inp: dict):
    return synth.widen(inp["Q"]), synth.widen(inp["K"]), synth.widen(inp["V"])


def nh_rows(wl, rows):
    return np.minimum((wl.q_offset + np.asarray(rows)) // wl.block_size, wl.n_blocks)


def r2_check(sel_gpu: np.ndarray, S64: np.ndarray, wl, rows):
    """sel_gpu [Hkv][nrows][Ks] (ascending, -1 padded) against fp64 scores
    S64 [Hkv][nrows][nblk].  Returns (n_rows_checked, n_swaps); asserts R2."""
    Ks = wl.k_blocks
    nh = nh_rows(wl, rows)
    swaps = 0
    for g in range(S64.shape[0]):
        for r in range(len(rows)):
            n = int(min(Ks, nh[r]))
            s = S64[g, r, :nh[r]]
            order = np.argsort(-s, kind="stable")
            ref = set(order[:n].tolist())
            got = [x for x in sel_gpu[g, r].tolist() if x >= 0]
            assert len(got) == n, (g, r, len(got), n)
            assert got == sorted(got)
            if n == 0:
                continue
            sk = s[order[n - 1]]
            tol = R2_TOL * max(1.0, abs(sk))
            diff = ref.symmetric_difference(got)
            for j in diff:
                assert abs(s[j] - sk) <= tol, (g, r, j, s[j], sk)
            swaps += len(diff) // 2
    return len(rows) * S64.shape[0], swaps


def clear_margin(S64: np.ndarray, wl, rows) -> np.ndarray:
    """[Hkv][nrows] bool: the fp64 selection is unambiguous under R2 (the
    k-th and (k+1)-th scores differ by more than twice the tolerance)."""
    Ks = wl.k_blocks
    nh = nh_rows(wl, rows)
    out = np.ones((S64.shape[0], len(rows)), bool)
    for g in range(S64.shape[0]):
        for r in range(len(rows)):
            if nh[r] <= Ks:
                continue
            s = np.sort(S64[g, r, :nh[r]])[::-1]
            tol = R2_TOL * max(1.0, abs(s[Ks - 1]))
            out[g, r] = (s[Ks - 1] - s[Ks]) > 2 * tol
    return out


def lse_bound_fp32_io(wl, Q: np.ndarray, K: np.ndarray, rows) -> np.ndarray:
    """[nrows][H] bound on |lse - lse64| when fp32 Q and K are rounded to bf16
    for the tensor cores: each logit moves by at most
    scale * (2 * 2^-9 + 2^-18) * sum_i |q_i k_i| (round-to-nearest on both
    factors), and the log-sum-exp moves by at most the largest logit change.
    The maximum runs over every causal key, a superset of the attended ones.
    A 1e-5 floor covers fp32 accumulation."""
    G = wl.n_q_heads // wl.n_kv_heads
    rows = np.asarray(rows)
    q = np.abs(Q[rows].astype(np.float64))                       # [n][H][d]
    k = np.abs(K.astype(np.float64))                             # [Tkv][Hkv][d]
    out = np.empty((len(rows), wl.n_q_heads))
    for h in range(wl.n_q_heads):
        a = q[:, h, :] @ k[:, h // G, :].T                       # [n][Tkv]
        causal = np.arange(K.shape[0])[None, :] <= (wl.q_offset + rows)[:, None]
        out[:, h] = np.where(causal, a, 0).max(1)
    return default_scale(wl) * (2.0 ** -8 + 2.0 ** -18) * out + 1e-5


def r3_check(O_gpu: np.ndarray, lse_gpu: np.ndarray, O64: np.ndarray, lse64: np.ndarray,
             row_mask=None, lse_tol=R3_LSE):
    """O_* [nrows][H][d], lse_* [H][nrows].  row_mask [nrows][H] selects the
    compared (row, head) pairs.  lse_tol: scalar, or [nrows][H] per pair."""
    dO = np.abs(O_gpu.astype(np.float64) - O64)
    dl = np.abs(lse_gpu.astype(np.float64) - lse64).T
    tol = np.broadcast_to(np.asarray(lse_tol, np.float64), dl.shape)
    if row_mask is not None:
        dO = dO[row_mask]
        dl = dl[row_mask]
        tol = tol[row_mask]
    assert dO.size > 0
    assert np.isfinite(dO).all() and np.isfinite(dl).all()
    assert dO.max() <= R3_MAX, dO.max()
    assert dO.mean() <= R3_MEAN, dO.mean()
    assert (dl <= tol).all(), float((dl / tol).max())
    return float(dO.max()), float(dO.mean()), float(dl.max())


def lse_tol_for(wl, inp, rows):
    """R3's 1e-3 for bf16 inputs (exact in bf16); the rounding bound for fp32 inputs."""
    if wl.dtype == "bf16":
        return R3_LSE
    Q, K, _ = widened(inp)
    return np.maximum(R3_LSE, lse_bound_fp32_io(wl, Q, K, rows))


def sample_rows(T: int, W: int, n: int, seed: int = 0) -> np.ndarray:
    """Spread rows plus tile edges and the last (ragged) rows."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    for x in (0, 1, W - 1, W, T - 1, T - 2, T // 2, (T // W) * W - 1):
        if 0 <= x < T:
            pick.add(x)
    return np.array(sorted(pick), np.int32)


def default_scale(wl) -> float:
    return 1.0 / math.sqrt(wl.head_dim)
