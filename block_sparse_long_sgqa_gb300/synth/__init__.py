"""Seeded synthetic workloads for the block-wise Sparse GQA prefill path.

This module only draws and lays out random inputs.  It holds none of the
method's arithmetic, which is why both the CUDA path (through the benchmark
and the tests) and the CPU oracle may read what it produces.

Workloads follow the shapes of the Step 5 Preview pages ("Inside Step 5
Preview", section "Sparse GQA": B = 8 position blocks, k = 4096 selected
tokens, contexts up to 1M):

* ``normal``: Q, K, V i.i.d. N(0, 1).
* ``clustered``: 64 seeded unit directions per KV group; every position p has
  a topic c(p) that is constant over runs of geometric length (mean 64
  positions, the pages' premise that adjacent tokens are semantically
  similar).  K[p][g] = 2.1 * u[g][c(p)] + N(0, 1) noise, V ~ N(0, 1), and
  Q[t][h] = 2.1 * u[g(h)][c(pos(t))] + noise whose lanes follow a stationary
  AR(1) process along t (marginal N(0, 1), correlation ``rho_q`` between
  neighbours; ``rho_q = 0`` gives i.i.d. noise).  2.1 = 0.7 * 3.
* needles (the 128K workload): every (query tile, KV group) draws one random
  unit direction r and 16 distinct historical blocks (the planted needles);
  8 r is added to all of that group's query heads in the tile, and 2 r to
  every key of each of the 16 blocks (a block planted by several tiles
  carries the sum of their directions).  A needle block then scores about
  8 * 2 = 16 above what it would score otherwise, while another block's score
  moves by 8 r against its keys' random part (a standard deviation near 3 at
  128 dimensions, the same for every query of the tile), so planted blocks
  sit far above the k-th score and a correct selection finds them.  The
  larger share sits on the query side so that the keys, which every tile
  reads, stay close to the clustered distribution.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsgqa_synth.so")
_lib = None

STREAM_Q, STREAM_K, STREAM_V, STREAM_TOPIC, STREAM_DIRS = 1, 2, 3, 4, 5
STREAM_SIG, STREAM_NEEDLE, STREAM_PAGES = 6, 7, 8

TOPIC_AMP = 0.7 * 3.0
N_TOPICS = 64
TOPIC_MEAN_RUN = 64.0
NEEDLES_PER_TILE = 16
NEEDLE_KEY_WEIGHT = 2.0
NEEDLE_QUERY_WEIGHT = 8.0
DEFAULT_RHO_Q = 0.99


def build(verbose: bool = False) -> str:
    """Compile the generator with the host C compiler (no CUDA involved)."""
    import subprocess

    src = os.path.join(_HERE, "synth.c")
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
    u64, i64, i32, f32, f64, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_float, ctypes.c_double, ctypes.c_void_p)
    lib.synth_fill_normal.argtypes = [u64, u64, i64, vp]
    lib.synth_fill_uniform.argtypes = [u64, u64, i64, vp]
    lib.synth_unit_dirs.argtypes = [u64, u64, i64, i32, vp]
    lib.synth_topic_runs.argtypes = [u64, u64, i64, f64, i32, vp]
    lib.synth_to_bf16.argtypes = [vp, i64, vp]
    lib.synth_clustered.argtypes = [u64, u64, i64, i32, i32, i32, i64, vp, vp, i32, f32, f64,
                                    vp, i64, f32, i32, vp]
    for f in (lib.synth_fill_normal, lib.synth_fill_uniform, lib.synth_unit_dirs,
              lib.synth_topic_runs, lib.synth_to_bf16, lib.synth_clustered):
        f.restype = None
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load().synth_fill_normal(seed, stream, n, _ptr(out))
    return out


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float64)
    _load().synth_fill_uniform(seed, stream, n, _ptr(out))
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().synth_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seq_q: int
    seq_kv: int
    q_offset: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    topk_tokens: int
    tile_q: int
    dtype: str            # "bf16" | "f32"
    dist: str             # "normal" | "clustered"
    needles: int = 0      # planted needle blocks per (query tile, group)
    page_size: int = 0    # 0: contiguous KV
    seed: int = 0
    rho_q: float = DEFAULT_RHO_Q

    @property
    def n_blocks(self) -> int:
        return self.seq_kv // self.block_size

    @property
    def k_blocks(self) -> int:
        return self.topk_tokens // self.block_size

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: seeds are 20261200 + workload number.
WORKLOADS = {
    "tiny_2k": Workload("tiny_2k", 2048, 2048, 0, 4, 1, 64, 8, 256, 16, "f32", "normal",
                        seed=20261201),
    "gqa_32k": Workload("gqa_32k", 32768, 32768, 0, 32, 4, 128, 8, 2048, 64, "bf16",
                        "clustered", seed=20261202),
    "step5_128k": Workload("step5_128k", 131072, 131072, 0, 64, 8, 128, 8, 4096, 64, "bf16",
                           "clustered", needles=NEEDLES_PER_TILE, seed=20261203),
    "sweep_64k_b1": Workload("sweep_64k_b1", 65536, 65536, 0, 32, 4, 128, 1, 2048, 64, "bf16",
                             "clustered", seed=20261204),
    "sweep_64k_b4": Workload("sweep_64k_b4", 65536, 65536, 0, 32, 4, 128, 4, 4096, 64, "bf16",
                             "clustered", seed=20261204),
    "sweep_64k_b8": Workload("sweep_64k_b8", 65536, 65536, 0, 32, 4, 128, 8, 4096, 64, "bf16",
                             "clustered", seed=20261204),
    "chunk_1m": Workload("chunk_1m", 8192, 1048576, 1048576 - 8192, 64, 8, 128, 8, 4096, 64,
                         "bf16", "clustered", page_size=64, seed=20261205),
}


def _choose_distinct(seed: int, stream: int, salt: int, n_range: int, k: int) -> np.ndarray:
    """k distinct integers from [0, n_range), drawn by a counter-based stream
    (Floyd's sampling); fewer when n_range < k."""
    k = min(k, n_range)
    u = uniform(seed, stream * 1000003 + salt, max(k, 1))
    chosen = []
    seen = set()
    for i, j in enumerate(range(n_range - k, n_range)):
        r = int(u[i] * (j + 1))
        r = min(r, j)
        if r in seen:
            r = j
        seen.add(r)
        chosen.append(r)
    return np.array(sorted(chosen), np.int32)


def make_inputs(wl: Workload, rho_q: Optional[float] = None) -> dict:
    """Generate Q [T][H][d], K and V [Tkv][Hkv][d] (bf16 bit patterns as uint16,
    or fp32), the topic labels, planted needles and the page table."""
    lib = _load()
    rho = wl.rho_q if rho_q is None else rho_q
    T, Tkv, H, Hkv, d, B = wl.seq_q, wl.seq_kv, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.block_size
    G = H // Hkv
    bf16 = wl.dtype == "bf16"
    edt = np.uint16 if bf16 else np.float32
    seed = wl.seed
    out: dict = {"workload": wl}

    topic = dirs = None
    if wl.dist == "clustered":
        topic = np.empty(Tkv, np.int32)
        lib.synth_topic_runs(seed, STREAM_TOPIC, Tkv, TOPIC_MEAN_RUN, N_TOPICS, _ptr(topic))
        dirs = np.empty((Hkv, N_TOPICS, d), np.float32)
        lib.synth_unit_dirs(seed, STREAM_DIRS, Hkv * N_TOPICS, d, _ptr(dirs))
        out["topic"] = topic
    elif wl.dist != "normal":
        raise ValueError(wl.dist)

    key_add = q_add = None
    if wl.needles:
        ntiles = (T + wl.tile_q - 1) // wl.tile_q
        tdir = np.empty((ntiles, Hkv, d), np.float32)  # one direction per (tile, group)
        lib.synth_unit_dirs(seed, STREAM_SIG, ntiles * Hkv, d, _ptr(tdir))
        key_add = np.zeros((-(-Tkv // B), Hkv, d), np.float32)  # [block][group][d], tail included
        needles = np.full((ntiles, Hkv, wl.needles), -1, np.int32)
        for tau in range(ntiles):
            nh = (wl.q_offset + tau * wl.tile_q) // B
            for g in range(Hkv):
                js = _choose_distinct(seed, STREAM_NEEDLE, tau * Hkv + g, nh, wl.needles)
                needles[tau, g, :len(js)] = js
                key_add[js, g] += tdir[tau, g]
        q_add = tdir
        out["needles"] = needles

    K = np.empty((Tkv, Hkv, d), edt)
    lib.synth_clustered(seed, STREAM_K, Tkv, Hkv, 1, d, 0, _ptr(topic), _ptr(dirs), N_TOPICS,
                        TOPIC_AMP, 0.0, _ptr(key_add), B, NEEDLE_KEY_WEIGHT, int(bf16), _ptr(K))
    V = np.empty((Tkv, Hkv, d), edt)
    lib.synth_clustered(seed, STREAM_V, Tkv, Hkv, 1, d, 0, None, None, N_TOPICS, 0.0, 0.0,
                        None, 1, 0.0, int(bf16), _ptr(V))
    Q = np.empty((T, H, d), edt)
    lib.synth_clustered(seed, STREAM_Q, T, H, G, d, wl.q_offset, _ptr(topic), _ptr(dirs),
                        N_TOPICS, TOPIC_AMP, rho if wl.dist == "clustered" else 0.0,
                        _ptr(q_add), wl.tile_q, NEEDLE_QUERY_WEIGHT, int(bf16), _ptr(Q))
    out.update(Q=Q, K=K, V=V)

    if wl.page_size:
        npages = -(-Tkv // wl.page_size)  # a partial last page counts
        u = uniform(seed, STREAM_PAGES, npages)
        out["page_table"] = np.argsort(u, kind="stable").astype(np.int32)
    return out


def to_paged(x: np.ndarray, page_table: np.ndarray, page_size: int) -> np.ndarray:
    """Lay a logical [Tkv][Hkv][d] tensor out as physical pages
    [npages][Hkv][page_size][d]: logical page i lives at physical page
    page_table[i]; a partial last page is padded with zeros."""
    Tkv, Hkv, d = x.shape
    npages = -(-Tkv // page_size)
    if npages * page_size != Tkv:
        x = np.concatenate([x, np.zeros((npages * page_size - Tkv, Hkv, d), x.dtype)])
    logical = x.reshape(npages, page_size, Hkv, d).transpose(0, 2, 1, 3)
    phys = np.empty_like(logical)
    phys[page_table] = logical
    return np.ascontiguousarray(phys)


def widen(x: np.ndarray) -> np.ndarray:
    """fp32 view of an input tensor (bf16 bit patterns are widened exactly)."""
    return bf16_bits_to_f32(x) if x.dtype == np.uint16 else np.ascontiguousarray(x, np.float32)
