"""sgqa_topk_union_noalloc: the top-k + union step for callers that cannot
allocate device memory (its selection scratch is a fixed array inside the
library).  Checked through the C ABI against sgqa_topk_union, which uses a
caller-provided workspace: the union outputs must be identical (selection
and union are exact integer work), on two calls in a row so that a stale
scratch array from the first call cannot hide a missing initialisation.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_long_sgqa_gb300 import synth

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["gqa_32k"].replace(name="noalloc", seq_q=700, seq_kv=830, q_offset=130,
                                        topk_tokens=256)


def _scores(seed):
    """Synthetic fp32 score matrices with the causal -inf pattern and frequent ties."""
    rng = np.random.default_rng(seed)
    S = rng.integers(-50, 50, size=(WL.n_kv_heads, WL.seq_q, WL.n_blocks)).astype(np.float32) / 8
    nh = np.minimum((WL.q_offset + np.arange(WL.seq_q)) // WL.block_size, WL.n_blocks)
    S[:, np.arange(WL.n_blocks)[None, :] >= nh[:, None]] = -np.inf
    return torch.from_numpy(S).cuda()


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


def test_noalloc_rejects_oversize_before_launch():
    from block_sparse_long_sgqa_gb300 import sgqa as s

    big = WL.replace(seq_q=4096, seq_kv=4096, q_offset=0, topk_tokens=8 * 1024, n_kv_heads=4,
                     n_q_heads=32)   # 4 * 4096 * 1024 entries > 2^21
    p = s.params_for(big)
    vp = ctypes.c_void_p
    rc = s._lib.sgqa_topk_union_noalloc(ctypes.byref(p), vp(0x1000), 0, big.seq_q, vp(0x1000),
                                        vp(0x1000), vp(0x1000), vp(0x1000), 1 << 40, None, None)
    assert rc == s.ERR_WORKSPACE
