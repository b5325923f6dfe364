"""ctypes binding of libsgqa.so (C ABI in include/sgqa.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (device memory and streams come from
torch); they are passed to the library as raw pointers.  Importing this module
fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsgqa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA = 0, 1, 2, 3, 4, 5
ERR_CAPACITY, ERR_TIMEOUT, ERR_BOUNDS = 6, 7, 8
BF16, FP32 = 0, 1
UNION_MASKED, UNION_FULL = 0, 1
INDEX_SPLIT, INDEX_BF16 = 0, 1
WS_INDEX_SCORES, WS_TOPK_UNION, WS_SPARSE_ATTN, WS_PREFILL, WS_ATTN_BWD, WS_DECODE = 1, 2, 3, 4, 5, 6
DEBUG_STALL = 0x5354414C  # SGQA_DEBUG_STALL: written into word 3 of a status buffer

EXPORTED = ("sgqa_workspace_bytes", "sgqa_union_capacity", "sgqa_block_merge", "sgqa_index_scores",
            "sgqa_topk_union", "sgqa_topk_union_noalloc", "sgqa_sparse_attn_fwd",
            "sgqa_sparse_attn_bwd", "sgqa_prefill", "sgqa_decode",
            "sgqa_prefill_ex", "sgqa_prefill_plan",
            "sgqa_set_launch_log", "sgqa_reset_status", "sgqa_read_status", "sgqa_status_string",
            "sgqa_version")
(K_MERGE, K_SPLIT, K_INDEX_QUERY, K_INDEX_SCORES, K_TOPK_UNION, K_ATTN, K_STAGE, K_TILE_UNION,
 K_SAMPLE_SCORES, K_ROW_TAU, K_ATTN_BWD) = (1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11)
KERNEL_NAMES = {1: "merge", 2: "split", 3: "index_query", 4: "index_scores", 5: "topk_union",
                6: "sparse_attn", 7: "stage_bf16", 8: "tile_union", 9: "sample_scores",
                10: "row_tau", 11: "sparse_attn_bwd"}


class Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "seq_q", "seq_kv", "q_offset", "n_q_heads", "n_kv_heads", "head_dim", "block_size",
        "topk_tokens", "tile_q", "page_size", "dtype", "union_mode")] + [
        ("softmax_scale", ctypes.c_float), ("batch", ctypes.c_int32),
        ("index_mode", ctypes.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class IndexInputs(ctypes.Structure):
    _fields_ = [("Qidx", ctypes.c_void_p), ("Kidx", ctypes.c_void_p)]


class BlockKeyCache(ctypes.Structure):
    _fields_ = [("Kbar", ctypes.c_void_p), ("Ksplit", ctypes.c_void_p),
                ("cap_blocks", ctypes.c_int32), ("valid_blocks", ctypes.c_int32)]


class LaunchLog(ctypes.Structure):
    _fields_ = [("capacity", ctypes.c_int32), ("count", ctypes.c_int32),
                ("start", ctypes.POINTER(ctypes.c_void_p)), ("stop", ctypes.POINTER(ctypes.c_void_p)),
                ("kind", ctypes.POINTER(ctypes.c_int32))]


class SgqaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_P = ctypes.POINTER(Params)
_lib.sgqa_workspace_bytes.argtypes = [_P, ctypes.c_int]
_lib.sgqa_workspace_bytes.restype = _sz
_lib.sgqa_union_capacity.argtypes = [_P]
_lib.sgqa_union_capacity.restype = _i64
_lib.sgqa_block_merge.argtypes = [_P, _vp, _vp, _i32, _i32, _vp, _vp, _vp]
_lib.sgqa_index_scores.argtypes = [_P, _vp, _vp, _i32, _i32, _vp, _vp, _sz, _vp, _vp]
_lib.sgqa_topk_union.argtypes = [_P, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _sz, _vp, _vp]
_lib.sgqa_topk_union_noalloc.argtypes = [_P, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp]
_lib.sgqa_sparse_attn_fwd.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                      _vp, _vp]
_lib.sgqa_sparse_attn_bwd.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _vp, _sz, _vp, _vp]
_lib.sgqa_prefill.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp, _vp]
_lib.sgqa_prefill_ex.argtypes = [_P, _vp, _vp, _vp, ctypes.POINTER(IndexInputs), _vp, _vp, _i32,
                                 _vp, _vp, _vp, _sz, _vp, _vp]
_lib.sgqa_decode.argtypes = [_P, _vp, _vp, _vp, _vp, ctypes.POINTER(BlockKeyCache), _vp, _vp, _vp,
                             _sz, _vp, _vp]
_lib.sgqa_prefill_plan.argtypes = [_P, ctypes.POINTER(_i64), ctypes.POINTER(_i32)]
_lib.sgqa_set_launch_log.argtypes = [ctypes.POINTER(LaunchLog)]
_lib.sgqa_reset_status.argtypes = [_vp, _vp]
_lib.sgqa_read_status.argtypes = [_vp, ctypes.POINTER(_i32), _vp]
_lib.sgqa_status_string.argtypes = [ctypes.c_int]
_lib.sgqa_status_string.restype = ctypes.c_char_p
_lib.sgqa_version.restype = ctypes.c_int
for _f in ("sgqa_block_merge", "sgqa_index_scores", "sgqa_topk_union", "sgqa_topk_union_noalloc",
           "sgqa_sparse_attn_fwd", "sgqa_sparse_attn_bwd",
           "sgqa_prefill", "sgqa_prefill_ex", "sgqa_decode", "sgqa_prefill_plan", "sgqa_set_launch_log", "sgqa_reset_status",
           "sgqa_read_status"):
    getattr(_lib, _f).restype = ctypes.c_int


def params(seq_q, seq_kv, q_offset, n_q_heads, n_kv_heads, head_dim, block_size, topk_tokens,
           tile_q, page_size=0, dtype=BF16, union_mode=UNION_MASKED, softmax_scale=0.0,
           batch=1, index_mode=INDEX_SPLIT) -> Params:
    return Params(seq_q, seq_kv, q_offset, n_q_heads, n_kv_heads, head_dim, block_size,
                  topk_tokens, tile_q, page_size, dtype, union_mode, softmax_scale, batch,
                  index_mode)


def params_for(wl, union_mode=UNION_MASKED, batch=1, index_mode=INDEX_SPLIT) -> Params:
    """Params of a synth.Workload (batch sequences of its shape)."""
    return params(wl.seq_q, wl.seq_kv, wl.q_offset, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                  wl.block_size, wl.topk_tokens, wl.tile_q, wl.page_size,
                  BF16 if wl.dtype == "bf16" else FP32, union_mode, batch=batch,
                  index_mode=index_mode)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise SgqaError(rc, what)


def version() -> int:
    return _lib.sgqa_version()


def status_string(code: int) -> str:
    return _lib.sgqa_status_string(code).decode()


def workspace_bytes(p: Params, which: int) -> int:
    return int(_lib.sgqa_workspace_bytes(ctypes.byref(p), which))


def union_capacity(p: Params) -> int:
    return int(_lib.sgqa_union_capacity(ctypes.byref(p)))


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(4, dtype=torch.int32, device=device)


def reset_status(status: torch.Tensor, stream=None) -> None:
    _check(_lib.sgqa_reset_status(_ptr(status), _stream(stream)), "sgqa_reset_status")


def read_status(status: torch.Tensor, stream=None):
    """Synchronises the stream; returns (code, detail)."""
    det = _i32(0)
    code = _lib.sgqa_read_status(_ptr(status), ctypes.byref(det), _stream(stream))
    return int(code), int(det.value)


def sgqa_block_merge(p, K, Kbar, blk_begin=0, blk_end=None, page_table=None, status=None, stream=None):
    if blk_end is None:
        blk_end = p.seq_kv // p.block_size
    _check(_lib.sgqa_block_merge(ctypes.byref(p), _ptr(K), _ptr(page_table), blk_begin, blk_end,
                                 _ptr(Kbar), _ptr(status), _stream(stream)), "sgqa_block_merge")


def sgqa_index_scores(p, Q, Kbar, q_begin, q_end, scores, ws, status=None, stream=None):
    _check(_lib.sgqa_index_scores(ctypes.byref(p), _ptr(Q), _ptr(Kbar), q_begin, q_end, _ptr(scores),
                                  _ptr(ws), ws.numel() * ws.element_size(), _ptr(status),
                                  _stream(stream)), "sgqa_index_scores")


def sgqa_topk_union(p, scores, q_begin, q_end, topk_idx, union_off, union_len, union_blk, union_mask,
                    ws=None, status=None, stream=None):
    _check(_lib.sgqa_topk_union(ctypes.byref(p), _ptr(scores), q_begin, q_end, _ptr(topk_idx),
                                _ptr(union_off), _ptr(union_len), _ptr(union_blk), _ptr(union_mask),
                                union_blk.numel(), _ptr(ws),
                                0 if ws is None else ws.numel() * ws.element_size(), _ptr(status),
                                _stream(stream)), "sgqa_topk_union")


def sgqa_topk_union_noalloc(p, scores, q_begin, q_end, union_off, union_len, union_blk,
                            union_mask, status=None, stream=None):
    """Top-k + union with the library's fixed scratch array (no workspace)."""
    _check(_lib.sgqa_topk_union_noalloc(ctypes.byref(p), _ptr(scores), q_begin, q_end,
                                        _ptr(union_off), _ptr(union_len), _ptr(union_blk),
                                        _ptr(union_mask), union_blk.numel(), _ptr(status),
                                        _stream(stream)), "sgqa_topk_union_noalloc")


def sgqa_sparse_attn_fwd(p, Q, K, V, union_off, union_len, union_blk, union_mask, O, lse,
                         page_table=None, ws=None, status=None, stream=None):
    _check(_lib.sgqa_sparse_attn_fwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(page_table),
                                     _ptr(union_off), _ptr(union_len), _ptr(union_blk),
                                     _ptr(union_mask), _ptr(O), _ptr(lse), _ptr(ws),
                                     0 if ws is None else ws.numel() * ws.element_size(),
                                     _ptr(status), _stream(stream)), "sgqa_sparse_attn_fwd")


def sgqa_sparse_attn_bwd(p, Q, K, V, union_off, union_len, union_blk, union_mask, O, lse, dO,
                         dQ, dK, dV, ws, page_table=None, status=None, stream=None):
    """Gradients of the main-path attention: dQ [T][H][d], dK and dV [Tkv][Hkv][d], fp32."""
    _check(_lib.sgqa_sparse_attn_bwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(page_table),
                                     _ptr(union_off), _ptr(union_len), _ptr(union_blk),
                                     _ptr(union_mask), _ptr(O), _ptr(lse), _ptr(dO), _ptr(dQ),
                                     _ptr(dK), _ptr(dV), _ptr(ws), ws.numel() * ws.element_size(),
                                     _ptr(status), _stream(stream)), "sgqa_sparse_attn_bwd")


def sgqa_prefill(p, Q, K, V, Kbar, O, lse, ws, page_table=None, kbar_valid_blocks=0, status=None,
                 stream=None):
    _check(_lib.sgqa_prefill(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(page_table), _ptr(Kbar),
                             kbar_valid_blocks, _ptr(O), _ptr(lse), _ptr(ws),
                             ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
           "sgqa_prefill")


def sgqa_prefill_ex(p, Q, K, V, Kbar, O, lse, ws, Qidx=None, Kidx=None, page_table=None,
                    kbar_valid_blocks=0, status=None, stream=None):
    """sgqa_prefill with separate index queries [T][Hkv][d] and/or index keys (K's layout)."""
    idx = IndexInputs(None if Qidx is None else _ptr(Qidx).value,
                      None if Kidx is None else _ptr(Kidx).value)
    _check(_lib.sgqa_prefill_ex(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), ctypes.byref(idx),
                                _ptr(page_table), _ptr(Kbar), kbar_valid_blocks, _ptr(O), _ptr(lse),
                                _ptr(ws), ws.numel() * ws.element_size(), _ptr(status),
                                _stream(stream)), "sgqa_prefill_ex")


class KeyCache:
    """A persistent block-key cache for sgqa_decode (device tensors owned here):
    Kbar [(batch,) Hkv, cap_blocks, d] fp32 and its hi/lo split [(batch,) 2, Hkv,
    cap_blocks, d] bf16; valid_blocks follows the calls."""

    def __init__(self, p: Params, cap_blocks: int, device="cuda"):
        nb = p.batch if p.batch > 1 else 1
        lead = (nb,) if nb > 1 else ()
        self.Kbar = torch.zeros(lead + (p.n_kv_heads, cap_blocks, p.head_dim), dtype=torch.float32,
                                device=device)
        self.Ksplit = torch.zeros(lead + (2, p.n_kv_heads, cap_blocks, p.head_dim),
                                  dtype=torch.bfloat16, device=device)
        self.c = BlockKeyCache(self.Kbar.data_ptr(), self.Ksplit.data_ptr(), cap_blocks, 0)

    @property
    def valid_blocks(self) -> int:
        return self.c.valid_blocks


def sgqa_decode(p, Q, K, V, cache: KeyCache, O, lse, ws, page_table=None, status=None, stream=None):
    _check(_lib.sgqa_decode(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(page_table),
                            ctypes.byref(cache.c), _ptr(O), _ptr(lse), _ptr(ws),
                            ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
           "sgqa_decode")


def sgqa_prefill_plan(p):
    """(queries per chunk, kernel launches) of one sgqa_prefill call with an empty cache."""
    c, n = _i64(0), _i32(0)
    _check(_lib.sgqa_prefill_plan(ctypes.byref(p), ctypes.byref(c), ctypes.byref(n)),
           "sgqa_prefill_plan")
    return int(c.value), int(n.value)


class launch_log:
    """Context manager installing a launch log of `capacity` CUDA event pairs.
    After the block, .entries() gives (kind, milliseconds) per logged launch
    (call it after synchronising)."""

    def __init__(self, capacity: int):
        self.events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(capacity)]
        s = torch.cuda.current_stream()
        for a, b in self.events:   # force creation of the underlying cudaEvent_t
            a.record(s)
            b.record(s)
        torch.cuda.synchronize()
        self._start = (ctypes.c_void_p * capacity)(*[a.cuda_event for a, _ in self.events])
        self._stop = (ctypes.c_void_p * capacity)(*[b.cuda_event for _, b in self.events])
        self._kind = (ctypes.c_int32 * capacity)()
        self.log = LaunchLog(capacity, 0, self._start, self._stop, self._kind)

    def __enter__(self):
        _check(_lib.sgqa_set_launch_log(ctypes.byref(self.log)), "sgqa_set_launch_log")
        return self

    def __exit__(self, *exc):
        _lib.sgqa_set_launch_log(None)
        return False

    @property
    def count(self) -> int:
        return self.log.count

    def entries(self):
        return [(self._kind[i], self.events[i][0].elapsed_time(self.events[i][1]))
                for i in range(self.log.count)]


# --------------------------------------------------------------------------- helpers
def _odt(p: Params):
    return torch.bfloat16 if p.dtype == BF16 else torch.float32


def alloc_workspace(p: Params, which: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(workspace_bytes(p, which), 1), dtype=torch.uint8, device=device)


def _nb(p: Params) -> int:
    return p.batch if p.batch > 1 else 1


def _bshape(p: Params, *shape):
    """A per-sequence shape, with the outer batch dimension when batch > 1."""
    return (p.batch, *shape) if p.batch > 1 else shape


def alloc_union(p: Params, device="cuda"):
    """(union_off, union_len, union_blk, union_mask) sized for the whole call."""
    ntiles = (p.seq_q + p.tile_q - 1) // p.tile_q
    cap = max(union_capacity(p), 1)
    return (torch.zeros(_nb(p) * p.n_kv_heads * ntiles, dtype=torch.int64, device=device),
            torch.zeros(_nb(p) * p.n_kv_heads * ntiles, dtype=torch.int32, device=device),
            torch.zeros(cap, dtype=torch.int32, device=device),
            torch.zeros(cap, dtype=torch.int64, device=device))


def alloc_outputs(p: Params, device="cuda"):
    O = torch.empty(_bshape(p, p.seq_q, p.n_q_heads, p.head_dim), dtype=_odt(p), device=device)
    lse = torch.empty(_bshape(p, p.n_q_heads, p.seq_q), dtype=torch.float32, device=device)
    return O, lse


def kbar_empty(p: Params, device="cuda") -> torch.Tensor:
    return torch.zeros(_bshape(p, p.n_kv_heads, p.seq_kv // p.block_size, p.head_dim),
                       dtype=torch.float32, device=device)


def default_scale(p: Params) -> float:
    return p.softmax_scale if p.softmax_scale > 0 else 1.0 / math.sqrt(p.head_dim)
