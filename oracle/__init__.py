"""CPU ORACLE for the block-wise Sparse GQA prefill path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never calls it and shares no code with it.

Thin ctypes wrappers over ``sgqa_oracle.c``; every step is documented there
with the passage of "Inside Step 5 Preview" (StepFun blog, section "Sparse
GQA") that it follows.  All arithmetic is fp64 unless a function says
otherwise.  Inputs are fp32 arrays (bf16 inputs are widened exactly first).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(verbose: bool = False) -> str:
    src = os.path.join(_HERE, "sgqa_oracle.c")
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", _LIB_PATH, src, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.orc_merge_tree_f32.argtypes = [vp, i64, i32, i32, i32, i64, i64, vp]
    lib.orc_merge_f64.argtypes = [vp, i64, i32, i32, i32, vp]
    lib.orc_index_query.argtypes = [vp, i64, i32, i32, i32, vp, i64, vp]
    lib.orc_scores.argtypes = [vp, vp, i64, i32, i32, i32, i64, vp, i64, vp]
    lib.orc_scores_bf16.argtypes = [vp, vp, i64, i32, i32, i32, i64, vp, i64, vp]
    lib.orc_select.argtypes = [vp, i32, i64, i32, i32, i64, vp, i64, i64, vp]
    lib.orc_union.argtypes = [vp, i64, i32, i64, i32, i64, i64, vp, vp, vp]
    lib.orc_union.restype = i64
    lib.orc_sparse_attn.argtypes = [vp, vp, vp, i64, i64, i64, i32, i32, i32, i32, i32, vp, i64,
                                    vp, vp, i32, f64, vp, i64, vp, vp]
    lib.orc_dense_attn.argtypes = [vp, vp, vp, i64, i64, i64, i32, i32, i32, f64, vp, i64, vp, vp]
    lib.orc_sparse_attn_bwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, i32, i32,
                                        vp, i64, vp, vp, i32, f64, vp, i64, vp, vp, vp]
    _lib = lib
    return lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, np.float32)


def _rows(rows, T: int) -> np.ndarray:
    if rows is None:
        return np.arange(T, dtype=np.int32)
    return np.ascontiguousarray(rows, np.int32)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed ({rc})")


def merge_tree_f32(K: np.ndarray, B: int, blk_begin: int = 0, blk_end: Optional[int] = None) -> np.ndarray:
    """K [Tkv][Hkv][d] fp32 -> Kbar [Hkv][nblk][d] fp32 (fixed pairwise tree; blocks
    outside [blk_begin, blk_end) are NaN)."""
    K = _f32(K)
    Tkv, Hkv, d = K.shape
    nblk = Tkv // B
    blk_end = nblk if blk_end is None else blk_end
    out = np.full((Hkv, nblk, d), np.nan, np.float32)
    _check(_load().orc_merge_tree_f32(_p(K), Tkv, Hkv, d, B, blk_begin, blk_end, _p(out)), "merge")
    return out


def merge_f64(K: np.ndarray, B: int) -> np.ndarray:
    K = _f32(K)
    Tkv, Hkv, d = K.shape
    out = np.empty((Hkv, Tkv // B, d), np.float64)
    _check(_load().orc_merge_f64(_p(K), Tkv, Hkv, d, B, _p(out)), "merge_f64")
    return out


def index_query(Q: np.ndarray, Hkv: int, rows=None) -> np.ndarray:
    """Q [T][H][d] -> qt [nrows][Hkv][d] fp64 (mean of each group's heads)."""
    Q = _f32(Q)
    T, H, d = Q.shape
    r = _rows(rows, T)
    out = np.empty((len(r), Hkv, d), np.float64)
    _check(_load().orc_index_query(_p(Q), T, H, Hkv, d, _p(r), len(r), _p(out)), "index_query")
    return out


def scores(qt: np.ndarray, Kbar: np.ndarray, B: int, q_offset: int, rows) -> np.ndarray:
    """qt [nrows][Hkv][d], Kbar [Hkv][nblk][d] (fp64) -> S [Hkv][nrows][nblk] fp64,
    -inf where block j is not historical for the row."""
    qt = np.ascontiguousarray(qt, np.float64)
    Kbar = np.ascontiguousarray(Kbar, np.float64)
    Hkv, nblk, d = Kbar.shape
    r = np.ascontiguousarray(rows, np.int32)
    out = np.empty((Hkv, len(r), nblk), np.float64)
    _check(_load().orc_scores(_p(qt), _p(Kbar), nblk, Hkv, d, B, q_offset, _p(r), len(r), _p(out)),
           "scores")
    return out


def scores_bf16(qt32: np.ndarray, Kbar32: np.ndarray, B: int, q_offset: int, rows) -> np.ndarray:
    """The bf16 indexer: qt32 [nrows][Hkv][d] and Kbar32 [Hkv][nblk][d] (fp32) ->
    S [Hkv][nrows][nblk] fp32 holding bf16 values (operands and score rounded
    to bf16, the products summed exactly), -inf where block j is not historical."""
    qt32 = np.ascontiguousarray(qt32, np.float32)
    Kbar32 = np.ascontiguousarray(Kbar32, np.float32)
    Hkv, nblk, d = Kbar32.shape
    r = np.ascontiguousarray(rows, np.int32)
    out = np.empty((Hkv, len(r), nblk), np.float32)
    _check(_load().orc_scores_bf16(_p(qt32), _p(Kbar32), nblk, Hkv, d, B, q_offset, _p(r), len(r),
                                   _p(out)), "scores_bf16")
    return out


def select(S: np.ndarray, B: int, q_offset: int, rows, Ks: int) -> np.ndarray:
    """S [Hkv][nrows][nblk] (fp32 or fp64) -> selections [Hkv][nrows][Ks] int32
    (ascending, -1 padded)."""
    is64 = S.dtype == np.float64
    S = np.ascontiguousarray(S, np.float64 if is64 else np.float32)
    Hkv, nrows, nblk = S.shape
    r = np.ascontiguousarray(rows, np.int32)
    assert len(r) == nrows
    out = np.empty((Hkv, nrows, Ks), np.int32)
    _check(_load().orc_select(_p(S), int(is64), nblk, Hkv, B, q_offset, _p(r), nrows, Ks, _p(out)),
           "select")
    return out


def union(sel: np.ndarray, W: int, nblk: int):
    """sel [Hkv][T][Ks] -> (uoff [Hkv][ntiles+1], ublk, umask) exact CSR."""
    sel = np.ascontiguousarray(sel, np.int32)
    Hkv, T, Ks = sel.shape
    ntiles = (T + W - 1) // W
    cap = Hkv * ntiles * min(W * Ks, max(nblk, 1)) + 1
    uoff = np.empty((Hkv, ntiles + 1), np.int32)
    ublk = np.empty(cap, np.int32)
    umask = np.empty(cap, np.uint64)
    n = _load().orc_union(_p(sel), T, Hkv, Ks, W, nblk, cap, _p(uoff), _p(ublk), _p(umask))
    if n < 0:
        raise RuntimeError("oracle union failed")
    return uoff, ublk[:n].copy(), umask[:n].copy()


def sparse_attn(Q, K, V, q_offset: int, B: int, sel: Optional[np.ndarray], mode: int = 0,
                union_csr=None, W: int = 64, scale: Optional[float] = None, rows=None):
    """Main-path attention.  Q [T][H][d], K/V [Tkv][Hkv][d] (fp32), sel
    [Hkv][T][Ks] over ALL T queries.  Returns O [nrows][H][d], lse [H][nrows]
    (fp64)."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    T, H, d = Q.shape
    Tkv, Hkv, _ = K.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    r = _rows(rows, T)
    if sel is None:
        sel = np.full((Hkv, T, 1), -1, np.int32)
    sel = np.ascontiguousarray(sel, np.int32)
    Ks = sel.shape[2]
    uoff = ublk = None
    if mode == 1:
        uoff, ublk, _ = union_csr if union_csr is not None else union(sel, W, Tkv // B)
        uoff = np.ascontiguousarray(uoff, np.int32)
        ublk = np.ascontiguousarray(ublk, np.int32)
    O = np.empty((len(r), H, d), np.float64)
    lse = np.empty((H, len(r)), np.float64)
    _check(_load().orc_sparse_attn(_p(Q), _p(K), _p(V), T, Tkv, q_offset, H, Hkv, d, B, mode,
                                   _p(sel), Ks, _p(uoff), _p(ublk), W, scale, _p(r), len(r),
                                   _p(O), _p(lse)), "sparse_attn")
    return O, lse


def sparse_attn_bwd(Q, K, V, dO, q_offset: int, B: int, sel: Optional[np.ndarray], mode: int = 0,
                    union_csr=None, W: int = 64, scale: Optional[float] = None, rows=None):
    """Gradients of L = sum(dO * O) for the attention of sparse_attn (same
    arguments; dO [nrows][H][d]).  Returns dQ [nrows][H][d], dK and dV
    [Tkv][Hkv][d] (fp64)."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    T, H, d = Q.shape
    Tkv, Hkv, _ = K.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    r = _rows(rows, T)
    dO = np.ascontiguousarray(dO, np.float64)
    assert dO.shape == (len(r), H, d)
    if sel is None:
        sel = np.full((Hkv, T, 1), -1, np.int32)
    sel = np.ascontiguousarray(sel, np.int32)
    Ks = sel.shape[2]
    uoff = ublk = None
    if mode == 1:
        uoff, ublk, _ = union_csr if union_csr is not None else union(sel, W, Tkv // B)
        uoff = np.ascontiguousarray(uoff, np.int32)
        ublk = np.ascontiguousarray(ublk, np.int32)
    dQ = np.empty((len(r), H, d), np.float64)
    dK = np.empty((Tkv, Hkv, d), np.float64)
    dV = np.empty((Tkv, Hkv, d), np.float64)
    _check(_load().orc_sparse_attn_bwd(_p(Q), _p(K), _p(V), _p(dO), T, Tkv, q_offset, H, Hkv, d,
                                       B, mode, _p(sel), Ks, _p(uoff), _p(ublk), W, scale, _p(r),
                                       len(r), _p(dQ), _p(dK), _p(dV)), "sparse_attn_bwd")
    return dQ, dK, dV


def dense_attn(Q, K, V, q_offset: int, scale: Optional[float] = None, rows=None):
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    T, H, d = Q.shape
    Tkv, Hkv, _ = K.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    r = _rows(rows, T)
    O = np.empty((len(r), H, d), np.float64)
    lse = np.empty((H, len(r)), np.float64)
    _check(_load().orc_dense_attn(_p(Q), _p(K), _p(V), T, Tkv, q_offset, H, Hkv, d, scale, _p(r),
                                  len(r), _p(O), _p(lse)), "dense_attn")
    return O, lse


def prefill_rows(Q, K, V, q_offset: int, B: int, Ks: int, rows, scale=None, Qidx=None, Kidx=None):
    """Mode-A prefill for a subset of query rows, end to end in fp64: merge,
    index query, scores, top-k, attention.  Returns (S, sel_rows, O, lse) with
    S [Hkv][nrows][nblk], sel_rows [Hkv][nrows][Ks].  Qidx [T][Hkv][d] and Kidx
    (K's shape), when given, are the index queries and keys: the index query of
    group g is Qidx[t][g] itself and the block keys are Kidx's block means."""
    T, H, d = Q.shape
    Tkv, Hkv, _ = K.shape
    r = np.ascontiguousarray(rows, np.int32)
    Kbar = merge_f64(K if Kidx is None else Kidx, B)
    qt = index_query(Q if Qidx is None else Qidx, Hkv, r)
    S = scores(qt, Kbar, B, q_offset, r)
    sel_rows = select(S, B, q_offset, r, Ks)
    # scatter the rows' selections into a full-size table for the attention step
    sel = np.full((Hkv, T, Ks), -1, np.int32)
    sel[:, r, :] = sel_rows
    O, lse = sparse_attn(Q, K, V, q_offset, B, sel, 0, scale=scale, rows=r)
    return S, sel_rows, O, lse
