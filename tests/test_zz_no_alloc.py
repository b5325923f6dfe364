"""sgqa_topk_union_noalloc: the top-k + union step for callers that cannot
allocate device memory (its selection scratch is a fixed array inside the
library).  Checked through the C ABI against sgqa_topk_union, which uses a
caller-provided workspace, and against the CPU oracle's select and union on
the same fp32 scores: the union outputs must be identical (selection and
union are exact integer work), on two calls in a row so that a stale
scratch array from the first call cannot hide a missing initialisation.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["gqa_32k"].replace(name="noalloc", seq_q=700, seq_kv=830, q_offset=130,
                                        topk_tokens=256)


# Rows of 17500+ blocks (the CTA-per-row select, which also writes into the
# fixed array), one KV group, called on the second tile only (q_begin > 0).
WL_LONG = synth.WORKLOADS["gqa_32k"].replace(name="noalloc_long", seq_q=128, seq_kv=140128,
                                             q_offset=140000, n_q_heads=8, n_kv_heads=1,
                                             topk_tokens=37 * 8)


def _scores_np(seed, wl=WL, q_begin=0, q_end=None):
    """Synthetic fp32 score matrices of queries [q_begin, q_end) with the
    causal -inf pattern and frequent ties."""
    q_end = wl.seq_q if q_end is None else q_end
    rng = np.random.default_rng(seed)
    S = rng.integers(-50, 50, size=(wl.n_kv_heads, q_end - q_begin, wl.n_blocks)).astype(np.float32) / 8
    nh = np.minimum((wl.q_offset + np.arange(q_begin, q_end)) // wl.block_size, wl.n_blocks)
    S[:, np.arange(wl.n_blocks)[None, :] >= nh[:, None]] = -np.inf
    return S


def _scores(seed):
    return torch.from_numpy(_scores_np(seed)).cuda()


def _oracle_lists(S, wl, q_begin, q_end):
    """The oracle's union lists of the tiles of [q_begin, q_end), from the same fp32 scores."""
    rows = np.arange(q_begin, q_end, dtype=np.int32)
    sel = oracle.select(S, wl.block_size, wl.q_offset, rows, wl.k_blocks)
    uoff, ublk, umask = oracle.union(sel, wl.tile_q, wl.n_blocks)
    return [(ublk[uoff[g, t]:uoff[g, t + 1]].tolist(), umask[uoff[g, t]:uoff[g, t + 1]].tolist())
            for g in range(uoff.shape[0]) for t in range(uoff.shape[1] - 1)]


def _outputs(s, p):
    return s.alloc_union(p)


def _lists(uo, ul, ub, um):
    uo, ul, ub, um = (x.cpu().numpy() for x in (uo, ul, ub, um))
    return [(ub[o:o + n].tolist(), um[o:o + n].tolist()) for o, n in zip(uo, ul)]


def test_noalloc_matches_workspace_version_twice():
    from block_sparse_long_sgqa_gb300 import sgqa as s

    p = s.params_for(WL)
    ws = s.alloc_workspace(p, s.WS_TOPK_UNION)
    for seed in (1, 2):  # two calls in a row, different inputs
        scores = _scores(seed)
        ref = _outputs(s, p)
        st = s.new_status()
        s.sgqa_topk_union(p, scores, 0, WL.seq_q, None, *ref, ws=ws, status=st)
        assert s.read_status(st)[0] == 0
        got = _outputs(s, p)
        for x in got:          # poison the outputs: every compared word must be written
            x.fill_(-5)
        st2 = s.new_status()
        s.sgqa_topk_union_noalloc(p, scores, 0, WL.seq_q, *got, status=st2)
        assert s.read_status(st2)[0] == 0
        assert _lists(*got) == _lists(*ref)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        got_u = [(b, [m & (2**64 - 1) for m in ms]) for b, ms in _lists(*got)]
        assert got_u == _oracle_lists(scores.cpu().numpy(), WL, 0, WL.seq_q)


def test_noalloc_long_rows_second_tile_twice():
    """Rows of more than 16384 blocks, on a query range that starts at the
    second tile, against the workspace version and the oracle, twice."""
    from block_sparse_long_sgqa_gb300 import sgqa as s

    wl, qb, qe = WL_LONG, 64, 128
    p = s.params_for(wl)
    ws = s.alloc_workspace(p, s.WS_TOPK_UNION)
    ntiles = wl.seq_q // wl.tile_q
    for seed in (3, 4):
        S = _scores_np(seed, wl, qb, qe)
        scores = torch.from_numpy(S).cuda()
        ref = s.alloc_union(p)
        st = s.new_status()
        s.sgqa_topk_union(p, scores, qb, qe, None, *ref, ws=ws, status=st)
        assert s.read_status(st)[0] == 0
        got = s.alloc_union(p)
        for x in got:
            x.fill_(-5)
        st2 = s.new_status()
        s.sgqa_topk_union_noalloc(p, scores, qb, qe, *got, status=st2)
        assert s.read_status(st2)[0] == 0
        # tile 1 of the (single) group was written; compare it
        lst_got = _lists(*got)[1:ntiles]
        assert lst_got == _lists(*ref)[1:ntiles]
        got_u = [(b, [m & (2**64 - 1) for m in ms]) for b, ms in lst_got]
        assert got_u == _oracle_lists(S, wl, qb, qe)


def test_noalloc_rejects_oversize_before_launch():
    from block_sparse_long_sgqa_gb300 import sgqa as s

    big = WL.replace(seq_q=4096, seq_kv=4096, q_offset=0, topk_tokens=8 * 1024, n_kv_heads=4,
                     n_q_heads=32)   # 4 * 4096 * 1024 entries > 2^21
    p = s.params_for(big)
    vp = ctypes.c_void_p
    rc = s._lib.sgqa_topk_union_noalloc(ctypes.byref(p), vp(0x1000), 0, big.seq_q, vp(0x1000),
                                        vp(0x1000), vp(0x1000), vp(0x1000), 1 << 40, None, None)
    assert rc == s.ERR_WORKSPACE
