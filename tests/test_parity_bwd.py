"""GPU parity of the attention backward (sgqa_sparse_attn_bwd) against the
oracle's fp64 backward (orc_sparse_attn_bwd, pinned in test_oracle_pins.py by
finite differences, autograd on the dense case and invariants).

The GPU backward is fed what a training step has: the GPU forward's O (bf16)
and log-sum-exp on the same block lists, and a seeded upstream gradient dO.
Its tensor cores see bf16 operands (Q, K, V, dO, and P and dS rounded to bf16
for the products), so its error against fp64 is bounded like the forward's:
max-abs within 2.5e-2 and mean-abs within 2.5e-3 of each gradient's largest
magnitude.  Results are deterministic (each gradient element is summed in one
place in a fixed order): two calls agree bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth
from helpers import dev_inputs, to_dev, widened
from test_parity_steps import SMALL, _upload_union, inputs

pytestmark = pytest.mark.gpu

CASES = ["b8", "b16", "w16_g8", "d64_g2", "paged", "needles", "few_b8", "few_b16_paged"]
TOL_MAX, TOL_MEAN = 2.5e-2, 2.5e-3


@pytest.fixture(scope="module")
def s():
    from block_sparse_long_sgqa_gb300 import sgqa

    return sgqa


def run_bwd(s, p, d, union, O, lse, dO, wl):
    dQ = torch.empty(wl.seq_q, wl.n_q_heads, wl.head_dim, device="cuda")
    dK = torch.full((wl.seq_kv, wl.n_kv_heads, wl.head_dim), float("nan"), device="cuda")
    dV = torch.full_like(dK, float("nan"))
    st = s.new_status()
    s.sgqa_sparse_attn_bwd(p, d["Q"], d["K"], d["V"], *union, O, lse, dO, dQ, dK, dV,
                           s.alloc_workspace(p, s.WS_ATTN_BWD), page_table=d["page_table"],
                           status=st)
    code, det = s.read_status(st)
    assert code == 0, (s.status_string(code), det)
    return dQ, dK, dV


def close(got, ref, name):
    got = got.double().cpu().numpy()
    scale = max(1e-30, float(np.abs(ref).max()))
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), name
    assert err.max() <= TOL_MAX * scale, (name, err.max() / scale)
    assert err.mean() <= TOL_MEAN * scale, (name, err.mean() / scale)
    return err.max() / scale, err.mean() / scale


@pytest.mark.parametrize("name", CASES)
@pytest.mark.parametrize("mode", [0, 1])
def test_attn_bwd_vs_oracle(s, name, mode):
    wl, inp = SMALL[name], inputs(name)
    p = s.params_for(wl, union_mode=mode)
    rows = np.arange(wl.seq_q, dtype=np.int32)
    Q, K, V = widened(inp)
    S = oracle.scores(oracle.index_query(Q, wl.n_kv_heads, rows), oracle.merge_f64(K, wl.block_size),
                      wl.block_size, wl.q_offset, rows)
    sel = oracle.select(S, wl.block_size, wl.q_offset, rows, wl.k_blocks)
    csr = oracle.union(sel, wl.tile_q, wl.n_blocks)
    d = dev_inputs(inp)
    union = _upload_union(*csr, wl.n_kv_heads, 0)
    O, lse = s.alloc_outputs(p)
    st = s.new_status()
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], *union, O, lse, page_table=d["page_table"],
                           ws=s.alloc_workspace(p, s.WS_SPARSE_ATTN), status=st)
    assert s.read_status(st)[0] == 0
    rng = np.random.default_rng(77)
    dOb = synth.to_bf16_bits(rng.standard_normal((wl.seq_q, wl.n_q_heads, wl.head_dim)).astype(np.float32))
    dO = to_dev(dOb)
    dQ, dK, dV = run_bwd(s, p, d, union, O, lse, dO, wl)
    dQ64, dK64, dV64 = oracle.sparse_attn_bwd(Q, K, V, synth.widen(dOb).astype(np.float64),
                                              wl.q_offset, wl.block_size, sel, mode, csr, wl.tile_q)
    close(dQ, dQ64, "dQ")
    close(dK, dK64, "dK")
    close(dV, dV64, "dV")
    # deterministic: a second call gives the same bits
    dQ2, dK2, dV2 = run_bwd(s, p, d, union, O, lse, dO, wl)
    assert torch.equal(dQ, dQ2) and torch.equal(dK, dK2) and torch.equal(dV, dV2)


def test_attn_bwd_rejects_unsupported(s):
    """B < 8 and fp32 inputs are rejected on the host before anything runs."""
    import ctypes

    vp = ctypes.c_void_p
    for wl in (SMALL["b4"], SMALL["tiny_2k"]):
        p = s.params_for(wl)
        args = [ctypes.byref(p)] + [vp(0x1000)] * 3 + [None] + [vp(0x1000)] * 11 + [1 << 40, None, None]
        assert s._lib.sgqa_sparse_attn_bwd(*args) == s.ERR_UNSUPPORTED


def whole_call_union(s, p, Q, Kbar, chunk=4096):
    """Union lists of every tile of the call, from the step entry points run
    on query ranges of `chunk` (a multiple of tile_q) so the scores stay small."""
    u = s.alloc_union(p)
    nblk = p.seq_kv // p.block_size
    ws = s.alloc_workspace(p, s.WS_TOPK_UNION)
    st = s.new_status()
    for q0 in range(0, p.seq_q, chunk):
        q1 = min(p.seq_q, q0 + chunk)
        sc = torch.empty(p.n_kv_heads, q1 - q0, nblk, device="cuda")
        s.sgqa_index_scores(p, Q, Kbar, q0, q1, sc, s.alloc_workspace(p, s.WS_INDEX_SCORES))
        s.sgqa_topk_union(p, sc, q0, q1, None, *u, ws=ws, status=st)
        del sc
    assert s.read_status(st)[0] == 0
    return u


def _tile_sel(u, wl, tau0, n):
    """The GPU union's per-query selections of queries [tau0 W, tau0 W + n)
    (whole tiles), as the oracle's [Hkv][n][Ks] table."""
    uo, ul, ub, um = u
    ntiles = (wl.seq_q + wl.tile_q - 1) // wl.tile_q
    W, Ks = wl.tile_q, wl.k_blocks
    sel = np.full((wl.n_kv_heads, n, Ks), -1, np.int32)
    for g in range(wl.n_kv_heads):
        for i in range(n):
            tau = tau0 + i // W
            o, ln = uo[g * ntiles + tau], ul[g * ntiles + tau]
            blks, masks = ub[o:o + ln], um[o:o + ln].view(np.uint64)
            mine = blks[((masks >> np.uint64(i % W)) & np.uint64(1)) == 1]
            sel[g, i, :len(mine)] = mine
    return sel


@pytest.mark.slow
@pytest.mark.parametrize("name", ["gqa_32k", "step5_128k"])
def test_attn_bwd_full_size(s, name):
    """The full workload: the GPU's own selection, forward and backward.
    Against the oracle: dQ of sampled tiles (each tile's queries as a
    sub-problem, their lists from the GPU union), and dK, dV of the last 128
    keys, which only the last 128 queries attend, so the oracle's backward of
    those queries alone gives them in full.  Over all keys, the identities
    sum_p dV_p = sum_rows dO and sum_p dK_p = 0 per group (a row's softmax
    weights sum to one) hold up to rounding.  Two calls are bit-identical."""
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    Kbar = s.kbar_empty(p)
    s.sgqa_block_merge(p, d["K"], Kbar)
    u = whole_call_union(s, p, d["Q"], Kbar)
    O, lse = s.alloc_outputs(p)
    st = s.new_status()
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], *u, O, lse,
                           ws=s.alloc_workspace(p, s.WS_SPARSE_ATTN), status=st)
    assert s.read_status(st)[0] == 0
    rng = np.random.default_rng(78)
    dOb = synth.to_bf16_bits(rng.standard_normal((wl.seq_q, wl.n_q_heads, wl.head_dim)).astype(np.float32))
    dO = to_dev(dOb)
    dQ, dK, dV = run_bwd(s, p, d, u, O, lse, dO, wl)
    # identities over every key and row
    G = wl.n_q_heads // wl.n_kv_heads
    sdO = dO.float().view(wl.seq_q, wl.n_kv_heads, G, wl.head_dim).double().sum((0, 2))
    rel_v = (dV.double().sum(0) - sdO).abs().max().item() / sdO.abs().max().item()
    rel_k = dK.double().sum(0).abs().max().item() / dK.double().abs().sum(0).max().item()
    assert rel_v < 1e-2 and rel_k < 1e-2, (rel_v, rel_k)
    # against the oracle
    Q, K, V = widened(inp)
    dOw = synth.widen(dOb).astype(np.float64)
    uh = tuple(x.cpu().numpy() for x in u)
    ntiles = (wl.seq_q + wl.tile_q - 1) // wl.tile_q
    W = wl.tile_q
    for tau in (0, ntiles // 3):
        q0 = tau * W
        n = min(W, wl.seq_q - q0)
        dQ64, _, _ = oracle.sparse_attn_bwd(Q[q0:q0 + n], K, V, dOw[q0:q0 + n], wl.q_offset + q0,
                                            wl.block_size, _tile_sel(uh, wl, tau, n), 0, W=W)
        close(dQ[q0:q0 + n], dQ64, f"dQ tile {tau}")
    q0 = wl.seq_q - 2 * W
    dQ64, dK64, dV64 = oracle.sparse_attn_bwd(Q[q0:], K, V, dOw[q0:], wl.q_offset + q0,
                                              wl.block_size, _tile_sel(uh, wl, q0 // W, 2 * W), 0, W=W)
    close(dQ[q0:], dQ64, "dQ last tiles")
    k0 = wl.seq_kv - 128
    close(dK[k0:], dK64[k0:], "dK last keys")
    close(dV[k0:], dV64[k0:], "dV last keys")
    dQ2, dK2, dV2 = run_bwd(s, p, d, u, O, lse, dO, wl)
    assert torch.equal(dQ, dQ2) and torch.equal(dK, dK2) and torch.equal(dV, dV2)


BWD_EDGE = {
    "one_query_at_0": SMALL["b8"].replace(name="be1", seq_q=1, seq_kv=1, q_offset=0),
    "under_one_block": SMALL["b8"].replace(name="be2", seq_q=5, seq_kv=5, q_offset=0),
    "ragged_one_query_tile": SMALL["b8"].replace(name="be3", seq_q=65, seq_kv=65, q_offset=0),
    "first_selection": SMALL["b8"].replace(name="be4", seq_q=2, seq_kv=271, q_offset=269),
}


@pytest.mark.parametrize("name", list(BWD_EDGE))
def test_attn_bwd_edge_shapes(s, name):
    """The backward on degenerate shapes (a single query with nothing before
    it, a call shorter than a block, a one-query last tile, rows just past
    k/B blocks) against the oracle's fp64 backward on the oracle's lists."""
    wl = BWD_EDGE[name]
    inp = synth.make_inputs(wl)
    p = s.params_for(wl)
    rows = np.arange(wl.seq_q, dtype=np.int32)
    Q, K, V = widened(inp)
    S = oracle.scores(oracle.index_query(Q, wl.n_kv_heads, rows), oracle.merge_f64(K, wl.block_size),
                      wl.block_size, wl.q_offset, rows)
    sel = oracle.select(S, wl.block_size, wl.q_offset, rows, wl.k_blocks)
    csr = oracle.union(sel, wl.tile_q, wl.n_blocks)
    d = dev_inputs(inp)
    union = _upload_union(*csr, wl.n_kv_heads, 0)
    O, lse = s.alloc_outputs(p)
    st = s.new_status()
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], *union, O, lse, page_table=d["page_table"],
                           ws=s.alloc_workspace(p, s.WS_SPARSE_ATTN), status=st)
    assert s.read_status(st)[0] == 0
    rng = np.random.default_rng(79)
    dOb = synth.to_bf16_bits(rng.standard_normal((wl.seq_q, wl.n_q_heads, wl.head_dim)).astype(np.float32))
    dQ, dK, dV = run_bwd(s, p, d, union, O, lse, to_dev(dOb), wl)
    dQ64, dK64, dV64 = oracle.sparse_attn_bwd(Q, K, V, synth.widen(dOb).astype(np.float64),
                                              wl.q_offset, wl.block_size, sel, 0, csr, wl.tile_q)
    for got, ref, nm in ((dQ, dQ64, "dQ"), (dK, dK64, "dK"), (dV, dV64, "dV")):
        if np.abs(ref).max() == 0.0:
            # a query that attends only itself has P = 1, so dS = dP - D = 0
            # and dQ, dK vanish exactly; the GPU's D comes from the bf16 O,
            # which leaves rounding noise
            assert np.abs(got.double().cpu().numpy()).max() <= 1e-4, nm
        else:
            close(got, ref, nm)
