"""Every workload at full size, in the launch configuration the benchmark
times, against the CPU oracle on sampled query tiles.

Per workload: the fused prefill (sgqa_prefill) runs over the whole workload
exactly as bench.py runs it (the 1M chunked prefill with its cached prefix
merged first).  Then, for a handful of tiles chosen at the first and last
tile, on both sides of every chunk boundary of the call, at the first row
that selects from threshold candidates and in between:

  R4  the block keys are bit-exact against the oracle's fp32 tree merge;
  R1  the tile's selection and union, computed by the step entry points on
      the GPU's own fp32 scores, are bit-exact against the oracle's select
      and union on those same scores;
  R2  that selection against the oracle's fp64 scores;
  R3  the GPU attention given the oracle's own (fp64) lists, on every row and
      head of the tile, and the fused output on the rows whose fp64 selection
      has a clear margin;
  and the fused output equals the step-by-step composition on the tile (the
  attention of the standalone lists), bit for bit.

Oracle cost is a few milliseconds per row on the host cores, so each workload
takes seconds beyond its input generation.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth
from helpers import clear_margin, dev_inputs, lse_tol_for, r2_check, r3_check, widened
from test_parity_steps import _gpu_union_lists, _oracle_union_lists, _upload_union

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

WORKLOADS = ["tiny_2k", "gqa_32k", "step5_128k", "sweep_64k_b1", "sweep_64k_b4", "sweep_64k_b8",
             "chunk_1m"]


@pytest.fixture(scope="module")
def s():
    from block_sparse_long_sgqa_gb300 import sgqa

    return sgqa


def sampled_tiles(wl, chunk: int, n_extra: int = 2, seed: int = 3):
    W, T = wl.tile_q, wl.seq_q
    ntiles = (T + W - 1) // W
    # the ends, and both sides of the first row with at least 2048 historical
    # blocks (where rows start to select from threshold candidates)
    must = {0, ntiles - 1}
    t_cand = 2048 * wl.block_size - wl.q_offset
    if 0 < t_cand < T:
        must.update({t_cand // W - 1, t_cand // W})
    # both sides of the chunk boundaries, a spread of at most six of them
    edges = sorted({x for c in range(chunk, T, chunk) for x in (c // W - 1, c // W)} | {ntiles // 2})
    if len(edges) > 6:
        edges = [edges[i] for i in np.linspace(0, len(edges) - 1, 6).round().astype(int)]
    pick = must | set(edges)
    rng = np.random.default_rng(seed)
    pick.update(rng.choice(ntiles, size=min(n_extra, ntiles), replace=False).tolist())
    return sorted(x for x in pick if 0 <= x < ntiles)


def run_full(s, wl, inp):
    """The benchmark's launch: device inputs, cached prefix merged first."""
    p = s.params_for(wl)
    d = dev_inputs(inp)
    Kbar = s.kbar_empty(p)
    kvalid = 0
    if wl.q_offset > 0:
        kvalid = wl.q_offset // wl.block_size
        s.sgqa_block_merge(p, d["K"], Kbar, 0, kvalid, page_table=d["page_table"])
    O, lse = s.alloc_outputs(p)
    ws = s.alloc_workspace(p, s.WS_PREFILL)
    st = s.new_status()
    s.sgqa_prefill(p, d["Q"], d["K"], d["V"], Kbar, O, lse, ws, page_table=d["page_table"],
                   kbar_valid_blocks=kvalid, status=st)
    code, det = s.read_status(st)
    assert code == 0, (s.status_string(code), det)
    del ws
    return p, d, Kbar, O, lse


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_vs_oracle(s, name):
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl)
    p, d, Kbar, O, lse = run_full(s, wl, inp)
    Q, K, V = widened(inp)
    B, W, Ks, nblk, Hkv = wl.block_size, wl.tile_q, wl.k_blocks, wl.n_blocks, wl.n_kv_heads

    # R4: the block keys, all of them (prefix merged by sgqa_block_merge, the
    # rest inside the prefill)
    ref_kbar = oracle.merge_tree_f32(K, B)
    assert np.array_equal(Kbar.cpu().numpy().view(np.uint32), ref_kbar.view(np.uint32))
    del ref_kbar

    chunk, _ = s.sgqa_prefill_plan(p)
    tiles = sampled_tiles(wl, chunk)
    Kbar64 = oracle.merge_f64(K, B)
    Og_all = O.float().cpu().numpy()
    lg_all = lse.cpu().numpy()
    lse_tol = None
    for tau in tiles:
        q0 = tau * W
        n = min(W, wl.seq_q - q0)
        rows = np.arange(q0, q0 + n, dtype=np.int32)
        sub = wl.replace(seq_q=n, q_offset=wl.q_offset + q0)
        ps = s.params_for(sub)
        Qs = d["Q"][q0:q0 + n].contiguous()

        # the step entry points on this tile (a call whose query 0 is the tile's first)
        scores = torch.empty(Hkv, n, nblk, device="cuda")
        s.sgqa_index_scores(ps, Qs, Kbar, 0, n, scores, s.alloc_workspace(ps, s.WS_INDEX_SCORES))
        sel = torch.empty(Hkv, n, Ks, dtype=torch.int32, device="cuda")
        uo, ul, ub, um = s.alloc_union(ps)
        st = s.new_status()
        s.sgqa_topk_union(ps, scores, 0, n, sel, uo, ul, ub, um, status=st)
        assert s.read_status(st)[0] == 0
        S32 = scores.cpu().numpy()
        del scores
        sel_g = sel.cpu().numpy()
        local = np.arange(n, dtype=np.int32)

        # R1 on the GPU's own fp32 scores
        ref_sel32 = oracle.select(S32, B, sub.q_offset, local, Ks)
        assert np.array_equal(sel_g, ref_sel32), ("R1 selection", tau)
        ref_u32 = oracle.union(ref_sel32, W, nblk)
        assert _gpu_union_lists(s, ps, uo, ul, ub, um) == _oracle_union_lists(*ref_u32), \
            ("R1 union", tau)
        del S32

        # R2 against the fp64 scores
        qt = oracle.index_query(Q, Hkv, rows)
        S64 = oracle.scores(qt, Kbar64, B, wl.q_offset, rows)
        r2_check(sel_g, S64, wl, rows)

        # R3: the GPU attention given the oracle's own lists, every row and head
        sel64 = oracle.select(S64, B, wl.q_offset, rows, Ks)
        Qt = Q[q0:q0 + n]
        O64, lse64 = oracle.sparse_attn(Qt, K, V, sub.q_offset, B, sel64, 0, W=W)
        uoff, ublk, umask = oracle.union(sel64, W, nblk)
        Ot, lt = s.alloc_outputs(ps)
        s.sgqa_sparse_attn_fwd(ps, Qs, d["K"], d["V"], *_upload_union(uoff, ublk, umask, Hkv, 0),
                               Ot, lt, page_table=d["page_table"],
                               ws=s.alloc_workspace(ps, s.WS_SPARSE_ATTN), status=st)
        assert s.read_status(st)[0] == 0
        if lse_tol is None or wl.dtype != "bf16":
            lse_tol = lse_tol_for(wl, inp, rows)
        r3_check(Ot.float().cpu().numpy(), lt.cpu().numpy(), O64, lse64, lse_tol=lse_tol)

        # R3 on the fused output, rows with a clear fp64 margin
        clear = clear_margin(S64, wl, rows)                       # [Hkv][n]
        G = wl.n_q_heads // Hkv
        mask = np.repeat(clear.T, G, axis=1)                      # [n][H]
        if mask.any():
            r3_check(Og_all[rows], lg_all[:, rows], O64, lse64, mask, lse_tol=lse_tol)

        # the fused output is the composition of the steps on this tile
        Oc, lc = s.alloc_outputs(ps)
        s.sgqa_sparse_attn_fwd(ps, Qs, d["K"], d["V"], uo, ul, ub, um, Oc, lc,
                               page_table=d["page_table"],
                               ws=s.alloc_workspace(ps, s.WS_SPARSE_ATTN), status=st)
        assert s.read_status(st)[0] == 0
        assert torch.equal(Oc, O[q0:q0 + n]), ("fused != composition (O)", tau)
        assert torch.equal(lc, lse[:, q0:q0 + n]), ("fused != composition (lse)", tau)
