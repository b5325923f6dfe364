"""GPU parity of the fused prefill (sgqa_prefill) against the CPU oracle.

End to end, the GPU's selection may legitimately differ from the fp64 oracle
at near-ties (rule R2), which changes the attention output of those rows; so
R3 is applied to the (row, head) pairs whose fp64 selection has a clear
margin, and R2 is checked on the standalone selection path that the fused
call is built from.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth
from helpers import clear_margin, dev_inputs, lse_tol_for, r2_check, r3_check, sample_rows, widened
from test_parity_steps import SMALL, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s():
    from block_sparse_long_sgqa_gb300 import sgqa

    return sgqa


def run_prefill(s, p, d, kbar=None, kvalid=0):
    O, lse = s.alloc_outputs(p)
    Kbar = s.kbar_empty(p) if kbar is None else kbar
    ws = s.alloc_workspace(p, s.WS_PREFILL)
    st = s.new_status()
    s.sgqa_prefill(p, d["Q"], d["K"], d["V"], Kbar, O, lse, ws, page_table=d["page_table"],
                   kbar_valid_blocks=kvalid, status=st)
    code, det = s.read_status(st)
    assert code == 0, (s.status_string(code), det)
    return O, lse, Kbar


def gpu_selection(s, p, d, Kbar, q_begin, q_end):
    """Standalone GPU path: index scores -> top-k (same kernels as the fused call)."""
    wl_T = q_end - q_begin
    nblk = p.seq_kv // p.block_size
    ws = s.alloc_workspace(p, s.WS_INDEX_SCORES)
    scores = torch.empty(p.n_kv_heads, wl_T, nblk, device="cuda")
    s.sgqa_index_scores(p, d["Q"], Kbar, q_begin, q_end, scores, ws)
    sel = torch.empty(p.n_kv_heads, wl_T, p.topk_tokens // p.block_size, dtype=torch.int32,
                      device="cuda")
    uo, ul, ub, um = s.alloc_union(p)
    st = s.new_status()
    s.sgqa_topk_union(p, scores, q_begin, q_end, sel, uo, ul, ub, um, status=st)
    assert s.read_status(st)[0] == 0
    return sel.cpu().numpy()


def check_end_to_end(s, wl, inp, O, lse, rows, Kbar, d):
    Q, K, V = widened(inp)
    S, sel_rows, O64, lse64 = oracle.prefill_rows(Q, K, V, wl.q_offset, wl.block_size, wl.k_blocks,
                                                  rows)
    clear = clear_margin(S, wl, rows)                       # [Hkv][nrows]
    G = wl.n_q_heads // wl.n_kv_heads
    mask = np.repeat(clear.T, G, axis=1)                    # [nrows][H]
    Og = O.float().cpu().numpy()[rows]
    lg = lse.cpu().numpy()[:, rows]
    stats = r3_check(Og, lg, O64, lse64, mask, lse_tol=lse_tol_for(wl, inp, rows))
    # R2 on the standalone selection of the same rows (contiguous query range)
    q0, q1 = int(rows.min()) // wl.tile_q * wl.tile_q, wl.seq_q
    q0 = min(q0, q1)
    sel = gpu_selection(s, s.params_for(wl), d, Kbar, q0, q1)
    r2_check(sel[:, rows - q0], S, wl, rows)
    return stats, float(mask.mean())


@pytest.mark.parametrize("name", list(SMALL))
def test_prefill_end_to_end(s, name):
    wl, inp = SMALL[name], inputs(name)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    O, lse, Kbar = run_prefill(s, p, d)
    rows = np.arange(wl.seq_q, dtype=np.int32)
    _, frac = check_end_to_end(s, wl, inp, O, lse, rows, Kbar, d)
    assert frac > 0.9


EDGE = {
    # one query at position 0: no historical block, only itself to attend
    "one_query_at_0": SMALL["b8"].replace(name="e1", seq_q=1, seq_kv=1, q_offset=0),
    # a call shorter than one block: every query sees only its own block
    "under_one_block": SMALL["b8"].replace(name="e2", seq_q=5, seq_kv=5, q_offset=0),
    # a last tile of one query, rows of at most nine blocks (all selected)
    "ragged_one_query_tile": SMALL["b8"].replace(name="e3", seq_q=65, seq_kv=65, q_offset=0),
    # one query at the first position of a block with exactly k/B blocks before it
    "block_start": SMALL["b8"].replace(name="e4", seq_q=1, seq_kv=257, q_offset=256),
    # one query whose row just exceeds k/B blocks (the first real selection)
    "first_selection": SMALL["b8"].replace(name="e5", seq_q=2, seq_kv=271, q_offset=269),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_prefill_edge_shapes(s, name):
    """Degenerate shapes through the fused call against the oracle: a single
    query with nothing before it, calls shorter than a block, a one-query
    last tile, and rows at the edge of the selection (exactly k/B blocks,
    one more)."""
    wl = EDGE[name]
    inp = synth.make_inputs(wl)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    O, lse, Kbar = run_prefill(s, p, d)
    assert torch.isfinite(O.float()).all() and torch.isfinite(lse).all()
    rows = np.arange(wl.seq_q, dtype=np.int32)
    if wl.seq_kv >= wl.block_size:  # R3 and R2 on the standalone selection
        _, frac = check_end_to_end(s, wl, inp, O, lse, rows, Kbar, d)
        assert frac >= 0.5
    else:  # no complete block: nothing to select, R3 on every row
        Q, K, V = widened(inp)
        S, _, O64, lse64 = oracle.prefill_rows(Q, K, V, wl.q_offset, wl.block_size, wl.k_blocks,
                                               rows)
        G = wl.n_q_heads // wl.n_kv_heads
        mask = np.repeat(clear_margin(S, wl, rows).T, G, axis=1)
        assert mask.all()
        r3_check(O.float().cpu().numpy()[rows], lse.cpu().numpy()[:, rows], O64, lse64, mask,
                 lse_tol=lse_tol_for(wl, inp, rows))


def test_prefill_mode_full(s):
    wl, inp = SMALL["b8"], inputs("b8")
    p = s.params_for(wl, union_mode=1)
    d = dev_inputs(inp)
    O, lse, _ = run_prefill(s, p, d)
    Q, K, V = widened(inp)
    rows = np.arange(wl.seq_q, dtype=np.int32)
    S = oracle.scores(oracle.index_query(Q, wl.n_kv_heads, rows), oracle.merge_f64(K, 8), 8,
                      wl.q_offset, rows)
    sel = oracle.select(S, 8, wl.q_offset, rows, wl.k_blocks)
    O64, lse64 = oracle.sparse_attn(Q, K, V, wl.q_offset, 8, sel, mode=1, W=wl.tile_q)
    # a near-tie anywhere in a tile can change that tile's union: compare tiles whose
    # rows all have a clear margin
    clear = clear_margin(S, wl, rows)
    tiles_ok = np.array([clear[:, i // wl.tile_q * wl.tile_q:(i // wl.tile_q + 1) * wl.tile_q].all()
                         for i in rows])
    G = wl.n_q_heads // wl.n_kv_heads
    mask = np.repeat(tiles_ok[:, None], wl.n_q_heads, axis=1)
    r3_check(O.float().cpu().numpy(), lse.cpu().numpy(), O64, lse64, mask)


def test_paged_equals_contiguous_bitexact(s):
    wl = SMALL["paged"]
    inp = inputs("paged")
    p = s.params_for(wl)
    O1, l1, _ = run_prefill(s, p, dev_inputs(inp))
    wl2 = wl.replace(page_size=0)
    p2 = s.params_for(wl2)
    inp2 = dict(inp, workload=wl2)
    O2, l2, _ = run_prefill(s, p2, dev_inputs(inp2))
    assert torch.equal(O1, O2) and torch.equal(l1, l2)


def test_chunked_prefill_bitexact(s):
    """Two calls (first half, then second half reusing the block-key cache)
    equal one call, bit for bit."""
    wl = SMALL["b8"]
    inp = inputs("b8")
    d = dev_inputs(inp)
    p = s.params_for(wl)
    O, lse, Kbar_full = run_prefill(s, p, d)
    half = (wl.seq_q // 2) // wl.tile_q * wl.tile_q
    # call 1: queries [0, half) with the KV prefix up to their last position
    wl1 = wl.replace(seq_q=half, seq_kv=wl.q_offset + half)
    p1 = s.params_for(wl1)
    d1 = dict(d, Q=d["Q"][:half].contiguous(), K=d["K"][:wl1.seq_kv].contiguous(),
              V=d["V"][:wl1.seq_kv].contiguous())
    O1, l1, Kb1 = run_prefill(s, p1, d1)
    # call 2: the rest, with the cached block keys of call 1
    wl2 = wl.replace(seq_q=wl.seq_q - half, q_offset=wl.q_offset + half)
    p2 = s.params_for(wl2)
    Kbar = s.kbar_empty(p2)
    Kbar[:, :Kb1.shape[1]] = Kb1
    d2 = dict(d, Q=d["Q"][half:].contiguous())
    O2, l2, Kb2 = run_prefill(s, p2, d2, kbar=Kbar, kvalid=Kb1.shape[1])
    assert torch.equal(Kb2, Kbar_full)
    assert torch.equal(torch.cat([O1, O2]), O)
    assert torch.equal(torch.cat([l1, l2], dim=1), lse)


@pytest.mark.parametrize("name", ["gqa_32k"])
def test_prefill_full_size_sampled(s, name):
    """The 32K workload at full size, in the launch configuration the benchmark
    times; sampled rows against the oracle."""
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    O, lse, Kbar = run_prefill(s, p, d)
    rows = sample_rows(wl.seq_q, wl.tile_q, 48, seed=1)
    rows = rows[rows >= wl.seq_q - 4096]  # one contiguous range for the standalone selection
    _, frac = check_end_to_end(s, wl, inp, O, lse, rows, Kbar, d)
    assert frac > 0.8


def composition(s, p, d, Kbar):
    """The fused prefill's steps called one by one through the C ABI: full
    score rows, the row select on them, the tile union and the attention."""
    nblk = p.seq_kv // p.block_size
    scores = torch.empty(p.n_kv_heads, p.seq_q, nblk, device="cuda")
    s.sgqa_index_scores(p, d["Q"], Kbar, 0, p.seq_q, scores, s.alloc_workspace(p, s.WS_INDEX_SCORES))
    sel = torch.empty(p.n_kv_heads, p.seq_q, p.topk_tokens // p.block_size, dtype=torch.int32,
                      device="cuda")
    uo, ul, ub, um = s.alloc_union(p)
    st = s.new_status()
    s.sgqa_topk_union(p, scores, 0, p.seq_q, sel, uo, ul, ub, um, status=st)
    O, lse = s.alloc_outputs(p)
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], uo, ul, ub, um, O, lse,
                           page_table=d["page_table"], ws=s.alloc_workspace(p, s.WS_SPARSE_ATTN),
                           status=st)
    assert s.read_status(st)[0] == 0
    return O, lse


# Rows of 2560 .. 2815 blocks: every row of the fused call selects from the
# indexer's threshold candidates.  "period61" repeats the block keys with a
# period of 61 blocks, so each score value occurs about 45 times and the k-th
# score is tied (the lowest-index rule decides); "period2" leaves two distinct
# scores, so the candidates overflow and every row falls back to its full
# score row.
FILT = synth.WORKLOADS["gqa_32k"].replace(name="filt", seq_q=2048, seq_kv=22528, q_offset=20480)


def periodic_keys(inp, period):
    K = inp["K"]
    pos = np.arange(K.shape[0])
    return dict(inp, K=np.ascontiguousarray(K[(pos // 8 % period) * 8 + pos % 8]))


@pytest.mark.parametrize("case", ["clustered", "period61", "period2", "gqa_32k", "long"])
def test_prefill_candidates_equal_full_select(s, case):
    """The fused prefill selects rows of 2048 .. 16384 blocks from threshold
    candidates; those lists must be the ones the full score rows give, so the
    fused output equals the step-by-step composition bit for bit.  "gqa_32k"
    has rows on both sides of 2048 blocks in one chunk; "long" is the last
    4096 queries of the 128K workload (rows of 15872 .. 16383 blocks)."""
    if case == "long":
        wl = synth.WORKLOADS["step5_128k"].replace(name="long", seq_q=4096, q_offset=131072 - 4096)
    else:
        wl = synth.WORKLOADS["gqa_32k"] if case == "gqa_32k" else FILT
    inp = synth.make_inputs(wl)
    if case.startswith("period"):
        inp = periodic_keys(inp, int(case[6:]))
    p = s.params_for(wl)
    d = dev_inputs(inp)
    O, lse, Kbar = run_prefill(s, p, d)
    O2, lse2 = composition(s, p, d, Kbar)
    assert torch.equal(O, O2)
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("case", ["b8", "filt", "mixed"])
def test_prefill_plan_counts_launches(s, case):
    """sgqa_prefill_plan's launch count is the number of kernels the call
    enqueues: chunks without candidates (b8), with them (filt), and several
    chunks in one call (the 128K shapes at 64K tokens: two chunks of 32768
    queries, the first with rows on both sides of 2048 blocks)."""
    mixed = synth.WORKLOADS["step5_128k"].replace(name="mixed", seq_q=65536, seq_kv=65536)
    wl = {"b8": SMALL["b8"], "filt": FILT, "mixed": mixed}[case]
    p = s.params_for(wl)
    _, planned = s.sgqa_prefill_plan(p)
    d = dev_inputs(synth.make_inputs(wl))
    log = s.launch_log(planned + 64)
    with log:
        run_prefill(s, p, d)
    assert log.count == planned


@pytest.mark.parametrize("pos", [20000, 150001])
def test_decode_step_paged(s, pos):
    """A decode step: one query at a position that ends mid-page, over a paged
    cache (64-token pages, the 1M workload's heads) whose earlier blocks' keys
    are cached; against the oracle.  At 20000 the row selects from threshold
    candidates, at 150001 (18750 blocks) it takes the CTA-per-row select."""
    wl = synth.WORKLOADS["chunk_1m"].replace(name="decode", seq_q=1, q_offset=pos, seq_kv=pos + 1)
    inp = synth.make_inputs(wl)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    kvalid = pos // wl.block_size  # blocks complete before this token
    Kbar = s.kbar_empty(p)
    s.sgqa_block_merge(p, d["K"], Kbar, 0, kvalid, page_table=d["page_table"])
    O, lse, Kbar = run_prefill(s, p, d, kbar=Kbar, kvalid=kvalid)
    rows = np.arange(1, dtype=np.int32)
    _, frac = check_end_to_end(s, wl, inp, O, lse, rows, Kbar, d)
    assert frac >= 0.5  # groups whose k-th score is a near-tie are checked by R2 only


def _batch2_inputs(s, paged):
    """Two sequences of one shape (different seeds) laid out for batch = 2: an
    outer dimension on Q, K and V, or one page pool shared by both with a
    page table per sequence."""
    base = SMALL["paged" if paged else "b8"]
    wls = [base, base.replace(seed=base.seed + 17)]
    inps = [synth.make_inputs(w) for w in wls]
    singles = [dev_inputs(i) for i in inps]
    d = {"Q": torch.stack([x["Q"] for x in singles])}
    if paged:
        npages = singles[0]["K"].shape[0]
        d["K"] = torch.cat([x["K"] for x in singles]).contiguous()
        d["V"] = torch.cat([x["V"] for x in singles]).contiguous()
        d["page_table"] = torch.stack([singles[0]["page_table"],
                                       singles[1]["page_table"] + npages]).contiguous()
    else:
        d["K"] = torch.stack([x["K"] for x in singles])
        d["V"] = torch.stack([x["V"] for x in singles])
        d["page_table"] = None
    return wls, inps, singles, d


@pytest.mark.parametrize("paged", [False, True])
def test_prefill_batch2_vs_single_calls_and_oracle(s, paged):
    """batch = 2 in one sgqa_prefill call: each sequence equals its own
    single-sequence call bit for bit and matches the oracle end to end."""
    wls, inps, singles, d = _batch2_inputs(s, paged)
    p2 = s.params_for(wls[0], batch=2)
    O, lse = s.alloc_outputs(p2)
    Kbar = s.kbar_empty(p2)
    st = s.new_status()
    s.sgqa_prefill(p2, d["Q"], d["K"], d["V"], Kbar, O, lse, s.alloc_workspace(p2, s.WS_PREFILL),
                   page_table=d["page_table"], status=st)
    assert s.read_status(st)[0] == 0
    p1 = s.params_for(wls[0])
    rows = np.arange(wls[0].seq_q, dtype=np.int32)
    for b in range(2):
        O1, l1, Kb1 = run_prefill(s, p1, singles[b])
        assert torch.equal(O[b], O1) and torch.equal(lse[b], l1) and torch.equal(Kbar[b], Kb1)
        _, frac = check_end_to_end(s, wls[b], inps[b], O[b], lse[b], rows, Kb1, singles[b])
        assert frac > 0.9


@pytest.mark.parametrize("paged", [False, True])
def test_steps_batch2_vs_single_calls(s, paged):
    """The step entry points with batch = 2 (merge, scores, top-k and union,
    attention, and the no-allocation top-k) equal single calls bit for bit."""
    wls, inps, singles, d = _batch2_inputs(s, paged)
    wl = wls[0]
    p2, p1 = s.params_for(wl, batch=2), s.params_for(wl)
    T, Hkv, nblk, Ks = wl.seq_q, wl.n_kv_heads, wl.n_blocks, wl.k_blocks
    st = s.new_status()
    Kbar = s.kbar_empty(p2)
    s.sgqa_block_merge(p2, d["K"], Kbar, page_table=d["page_table"], status=st)
    scores = torch.empty(2, Hkv, T, nblk, device="cuda")
    s.sgqa_index_scores(p2, d["Q"], Kbar, 0, T, scores, s.alloc_workspace(p2, s.WS_INDEX_SCORES))
    sel = torch.empty(2, Hkv, T, Ks, dtype=torch.int32, device="cuda")
    u2 = s.alloc_union(p2)
    s.sgqa_topk_union(p2, scores, 0, T, sel, *u2, status=st)
    un = s.alloc_union(p2)
    s.sgqa_topk_union_noalloc(p2, scores, 0, T, *un, status=st)
    O, lse = s.alloc_outputs(p2)
    s.sgqa_sparse_attn_fwd(p2, d["Q"], d["K"], d["V"], *u2, O, lse, page_table=d["page_table"],
                           ws=s.alloc_workspace(p2, s.WS_SPARSE_ATTN), status=st)
    assert s.read_status(st)[0] == 0
    cap1 = s.union_capacity(p1)
    ntl = Hkv * ((T + wl.tile_q - 1) // wl.tile_q)
    for b in range(2):
        x = singles[b]
        Kb1 = s.kbar_empty(p1)
        s.sgqa_block_merge(p1, x["K"], Kb1, page_table=x["page_table"])
        sc1 = torch.empty(Hkv, T, nblk, device="cuda")
        s.sgqa_index_scores(p1, x["Q"], Kb1, 0, T, sc1, s.alloc_workspace(p1, s.WS_INDEX_SCORES))
        sel1 = torch.empty(Hkv, T, Ks, dtype=torch.int32, device="cuda")
        u1 = s.alloc_union(p1)
        s.sgqa_topk_union(p1, sc1, 0, T, sel1, *u1, status=st)
        O1, l1 = s.alloc_outputs(p1)
        s.sgqa_sparse_attn_fwd(p1, x["Q"], x["K"], x["V"], *u1, O1, l1,
                               page_table=x["page_table"],
                               ws=s.alloc_workspace(p1, s.WS_SPARSE_ATTN), status=st)
        assert s.read_status(st)[0] == 0
        assert torch.equal(Kbar[b], Kb1)
        assert torch.equal(scores[b], sc1)
        assert torch.equal(sel[b], sel1)
        for u in (u2, un):   # offsets, lengths, then the slots of sequence b
            assert torch.equal(u[0][b * ntl:(b + 1) * ntl], u1[0])
            assert torch.equal(u[1][b * ntl:(b + 1) * ntl], u1[1])
            for k in (2, 3):
                a = u[k][b * cap1:(b + 1) * cap1]
                for o, n in zip(u1[0].tolist(), u1[1].tolist()):
                    assert torch.equal(a[o:o + n], u1[k][o:o + n])
        assert torch.equal(O[b], O1) and torch.equal(lse[b], l1)
