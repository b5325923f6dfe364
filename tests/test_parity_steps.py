"""GPU parity of each step of the path against the CPU oracle, through the C ABI.

Small workloads that still span several tiles, a ragged last tile and a
query offset that is not block aligned.  Rules R1-R3 are stated in helpers.py.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth
from helpers import (clear_margin, dev_inputs, lse_tol_for, nh_rows, r2_check, r3_check, to_dev,
                     widened)

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["gqa_32k"]
SMALL = {
    "tiny_2k": synth.WORKLOADS["tiny_2k"],
    "b8": BASE.replace(name="b8", seq_q=1000, seq_kv=1123, q_offset=123, topk_tokens=256),
    "b1": BASE.replace(name="b1", seq_q=600, seq_kv=700, q_offset=100, block_size=1, topk_tokens=64),
    "b4": BASE.replace(name="b4", seq_q=700, seq_kv=777, q_offset=77, block_size=4, topk_tokens=128),
    "b16": BASE.replace(name="b16", seq_q=700, seq_kv=900, q_offset=200, block_size=16,
                        topk_tokens=256),
    "w16_g8": BASE.replace(name="w16_g8", seq_q=500, seq_kv=600, q_offset=100, tile_q=16,
                           topk_tokens=128),
    "paged": BASE.replace(name="paged", seq_q=1000, seq_kv=1152, q_offset=152, page_size=64,
                          topk_tokens=256),
    "d64_g2": BASE.replace(name="d64_g2", seq_q=400, seq_kv=450, q_offset=50, n_q_heads=8,
                           n_kv_heads=4, head_dim=64, topk_tokens=96, tile_q=32),
    # key-by-key gathers (B < 8) from a paged cache with a partly filled last
    # page, and at head_dim 64
    "paged_b4": BASE.replace(name="paged_b4", seq_q=600, seq_kv=1000, q_offset=400, block_size=4,
                             page_size=64, topk_tokens=128),
    "d64_b2": BASE.replace(name="d64_b2", seq_q=300, seq_kv=380, q_offset=80, n_q_heads=8,
                           n_kv_heads=4, head_dim=64, block_size=2, topk_tokens=64, tile_q=32),
    # few queries over a longer cache: B >= 8 blocks gathered key by key
    # instead of copied from a packed cache (fewer selected blocks than cached)
    "few_b8": BASE.replace(name="few_b8", seq_q=8, seq_kv=3000, q_offset=2992, topk_tokens=256),
    "few_b16_paged": BASE.replace(name="few_b16_paged", seq_q=4, seq_kv=2000, q_offset=1996,
                                  head_dim=64, block_size=16, topk_tokens=256, page_size=64),
    # fp32 inputs over a paged cache, keys gathered: converted through the page table
    "f32_paged_b4": synth.WORKLOADS["tiny_2k"].replace(name="f32_paged_b4", seq_q=300, seq_kv=700,
                                                      q_offset=400, block_size=4, topk_tokens=64,
                                                      page_size=64),
    # degenerate: one query at position 0 (no block, no union) and a query
    # pair whose rows just exceed k/B blocks (the first real selection)
    "edge_one": BASE.replace(name="edge_one", seq_q=1, seq_kv=1, q_offset=0, topk_tokens=256),
    "edge_first_sel": BASE.replace(name="edge_first_sel", seq_q=2, seq_kv=271, q_offset=269,
                                   topk_tokens=256),
    # Step-5-shaped heads with planted needles: large logit jumps between stages
    # exercise the online-softmax rescale of O in TMEM
    "needles": synth.WORKLOADS["step5_128k"].replace(name="needles", seq_q=1200, seq_kv=1200,
                                                     topk_tokens=512),
}
_cache = {}


def inputs(name):
    if name not in _cache:
        _cache[name] = synth.make_inputs(SMALL[name])
    return _cache[name]


@pytest.fixture(scope="module")
def s():
    from block_sparse_long_sgqa_gb300 import sgqa

    assert torch.cuda.is_available()
    return sgqa


@pytest.mark.parametrize("name", list(SMALL))
def test_block_merge_bitexact(s, name):
    wl, inp = SMALL[name], inputs(name)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    st = s.new_status()
    Kbar = torch.full((wl.n_kv_heads, wl.n_blocks, wl.head_dim), float("nan"), device="cuda")
    s.sgqa_block_merge(p, d["K"], Kbar, page_table=d["page_table"], status=st)
    ref = oracle.merge_tree_f32(synth.widen(inp["K"]), wl.block_size)
    assert np.array_equal(Kbar.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # a sub-range leaves the other blocks untouched
    Kb2 = torch.full_like(Kbar, 7.0)
    nb = wl.n_blocks
    s.sgqa_block_merge(p, d["K"], Kb2, nb // 3, nb // 2, page_table=d["page_table"])
    got = Kb2.cpu().numpy()
    assert np.array_equal(got[:, nb // 3:nb // 2], ref[:, nb // 3:nb // 2])
    assert (got[:, :nb // 3] == 7.0).all() and (got[:, nb // 2:] == 7.0).all()
    assert s.read_status(st)[0] == 0


@pytest.mark.parametrize("name", ["tiny_2k", "b8", "b1", "b16", "d64_g2"])
def test_index_scores_accuracy(s, name):
    wl, inp = SMALL[name], inputs(name)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    Q, K, _ = widened(inp)
    Kbar = s.kbar_empty(p)
    s.sgqa_block_merge(p, d["K"], Kbar, page_table=d["page_table"])
    ws = s.alloc_workspace(p, s.WS_INDEX_SCORES)
    st = s.new_status()
    for qb, qe in ((0, wl.seq_q), (wl.seq_q // 3, wl.seq_q - 5)):
        scores = torch.empty(wl.n_kv_heads, qe - qb, wl.n_blocks, device="cuda")
        s.sgqa_index_scores(p, d["Q"], Kbar, qb, qe, scores, ws, status=st)
        got = scores.cpu().numpy().astype(np.float64)
        rows = np.arange(qb, qe)
        qt = oracle.index_query(Q, wl.n_kv_heads, rows)
        kb = oracle.merge_f64(K, wl.block_size)
        ref = oracle.scores(qt, kb, wl.block_size, wl.q_offset, rows)
        fin = np.isfinite(ref)
        assert np.array_equal(np.isfinite(got), fin)
        assert (got[~fin] == -np.inf).all()
        # the bf16 hi/lo split keeps every product within ~3 * 2^-18 of exact
        bound = np.einsum("rgi,gji->grj", np.abs(qt), np.abs(kb)) * 4e-5 + 1e-6
        err = np.abs(got[fin] - ref[fin])
        assert (err <= bound[fin]).all(), float((err / bound[fin]).max())
    assert s.read_status(st)[0] == 0


def _upload_union(uoff, ublk, umask, Hkv, ntiles):
    off = uoff[:, :-1].reshape(-1).astype(np.int64)
    ln = (uoff[:, 1:] - uoff[:, :-1]).reshape(-1).astype(np.int32)
    return (torch.from_numpy(off).cuda(), torch.from_numpy(ln).cuda(),
            torch.from_numpy(np.ascontiguousarray(ublk, np.int32)).cuda(),
            torch.from_numpy(np.ascontiguousarray(umask).view(np.int64)).cuda())


def _gpu_union_lists(s, p, uo, ul, ub, um):
    uo, ul, ub, um = (x.cpu().numpy() for x in (uo, ul, ub, um))
    return [(ub[o:o + n].tolist(), um[o:o + n].view(np.uint64).tolist()) for o, n in zip(uo, ul)]


def _oracle_union_lists(uoff, ublk, umask):
    out = []
    for g in range(uoff.shape[0]):
        for tau in range(uoff.shape[1] - 1):
            a, b = uoff[g, tau], uoff[g, tau + 1]
            out.append((ublk[a:b].tolist(), umask[a:b].tolist()))
    return out


def _fp32_scores_from_oracle(inp, wl, rows):
    Q, K, _ = widened(inp)
    S = oracle.scores(oracle.index_query(Q, wl.n_kv_heads, rows), oracle.merge_f64(K, wl.block_size),
                      wl.block_size, wl.q_offset, rows)
    return S.astype(np.float32)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("quant", [None, 0.5])
def test_topk_union_bitexact(s, name, quant):
    """R1: selection and union from the same fp32 scores are bit-exact.  quant
    rounds the scores to a coarse grid so that ties are everywhere."""
    wl, inp = SMALL[name], inputs(name)
    p = s.params_for(wl)
    rows = np.arange(wl.seq_q)
    S32 = _fp32_scores_from_oracle(inp, wl, rows)
    if quant:
        S32 = (np.round(S32 / quant) * quant).astype(np.float32)
    ref_sel = oracle.select(S32, wl.block_size, wl.q_offset, rows, wl.k_blocks)
    ref_u = oracle.union(ref_sel, wl.tile_q, wl.n_blocks)
    scores = torch.from_numpy(S32).cuda()
    sel = torch.full((wl.n_kv_heads, wl.seq_q, wl.k_blocks), -7, dtype=torch.int32, device="cuda")
    uo, ul, ub, um = s.alloc_union(p)
    st = s.new_status()
    s.sgqa_topk_union(p, scores, 0, wl.seq_q, sel, uo, ul, ub, um, status=st)
    assert s.read_status(st)[0] == 0
    assert np.array_equal(sel.cpu().numpy(), ref_sel)
    assert _gpu_union_lists(s, p, uo, ul, ub, um) == _oracle_union_lists(*ref_u)


@pytest.mark.parametrize("case", ["all_equal", "three_values", "neg_zero"])
def test_topk_union_degenerate_scores(s, case):
    """Rows longer than the bucket buffer with massive ties (the slow path),
    and signed zeros."""
    T, B, off, Hkv, Ks, W = 96, 8, 2600 * 8, 2, 100, 32
    wl = synth.Workload("deg", T, off + T, off, 8, Hkv, 128, B, Ks * B, W, "bf16", "normal")
    p = s.params_for(wl)
    rng = np.random.default_rng(5)
    shape = (Hkv, T, wl.n_blocks)
    if case == "all_equal":
        S32 = np.zeros(shape, np.float32)
    elif case == "three_values":
        S32 = rng.choice(np.array([-1.0, 0.25, 3.0], np.float32), size=shape)
    else:
        S32 = rng.choice(np.array([-0.0, 0.0, 1e-30, -1e-30], np.float32), size=shape)
    rows = np.arange(T)
    ref_sel = oracle.select(S32, B, off, rows, Ks)
    ref_u = oracle.union(ref_sel, W, wl.n_blocks)
    sel = torch.empty(Hkv, T, Ks, dtype=torch.int32, device="cuda")
    uo, ul, ub, um = s.alloc_union(p)
    st = s.new_status()
    s.sgqa_topk_union(p, torch.from_numpy(S32).cuda(), 0, T, sel, uo, ul, ub, um, status=st)
    assert s.read_status(st)[0] == 0
    assert np.array_equal(sel.cpu().numpy(), ref_sel)
    assert _gpu_union_lists(s, p, uo, ul, ub, um) == _oracle_union_lists(*ref_u)


@pytest.mark.parametrize("case", ["clustered", "clustered_ties", "iid", "sample_low", "sample_high"])
@pytest.mark.parametrize("Ks", [512, 37])
@pytest.mark.parametrize("kv_extra", [0, 80000])
def test_topk_union_long_rows(s, case, Ks, kv_extra):
    """Rows of 10000+ blocks, bit-exact against the oracle.  With kv_extra = 0
    the rows fit the shared-memory row kernel (threshold predicted from the
    previous row, else the exact radix select on the row); with a longer key
    range (20016 blocks) the warp-per-row kernel runs its candidate path (a
    sample of 8 in every 64 blocks, or the previous row, sets the threshold).
    Some scores are unrepresentative on purpose, so that candidates miss or
    overflow and rows fall back to the exact selects."""
    T, B, off, Hkv, W = 128, 8, 80000, 2, 64
    wl = synth.Workload("long", T, off + T + kv_extra, off, 8, Hkv, 128, B, Ks * B, W, "bf16",
                        "normal")
    p = s.params_for(wl)
    nb = wl.n_blocks
    rng = np.random.default_rng(11)
    # scores of clustered blocks: runs of 64 blocks share a level
    level = np.repeat(rng.normal(0.0, 1.0, (Hkv, 1, nb // 64 + 1)), 64, axis=2)[:, :, :nb]
    S = level + 0.3 * rng.normal(0.0, 1.0, (Hkv, T, nb))
    if case == "clustered_ties":
        S = np.round(S * 8.0) / 8.0
    elif case == "iid":
        S = rng.normal(0.0, 1.0, (Hkv, T, nb))
    elif case in ("sample_low", "sample_high"):
        sampled = (np.arange(nb) % 64) < 8
        S = rng.normal(0.0, 1.0, (Hkv, T, nb))
        S[:, :, sampled] += -6.0 if case == "sample_low" else 6.0
    S32 = np.ascontiguousarray(S, np.float32)
    rows = np.arange(T)
    ref_sel = oracle.select(S32, B, off, rows, Ks)
    ref_u = oracle.union(ref_sel, W, nb)
    sel = torch.empty(Hkv, T, Ks, dtype=torch.int32, device="cuda")
    uo, ul, ub, um = s.alloc_union(p)
    st = s.new_status()
    s.sgqa_topk_union(p, torch.from_numpy(S32).cuda(), 0, T, sel, uo, ul, ub, um, status=st)
    assert s.read_status(st)[0] == 0
    assert np.array_equal(sel.cpu().numpy(), ref_sel)
    assert _gpu_union_lists(s, p, uo, ul, ub, um) == _oracle_union_lists(*ref_u)


@pytest.mark.parametrize("case", ["clustered", "clustered_ties", "iid", "all_equal"])
@pytest.mark.parametrize("Ks", [37, 512, 2048])
def test_topk_union_cta_rows(s, case, Ks):
    """Rows of more than 16384 blocks (25000-25016 here) take the CTA-per-row
    select; bit-exact against the oracle.  "all_equal" puts every key in one
    bucket, too many for shared memory, so each digit level passes over the
    row again and the lowest indices win the tie."""
    T, B, off, Hkv, W = 128, 8, 200000, 2, 64
    wl = synth.Workload("cta", T, off + T, off, 8, Hkv, 128, B, Ks * B, W, "bf16", "normal")
    p = s.params_for(wl)
    nb = wl.n_blocks
    rng = np.random.default_rng(12)
    level = np.repeat(rng.normal(0.0, 1.0, (Hkv, 1, nb // 64 + 1)), 64, axis=2)[:, :, :nb]
    S = level + 0.3 * rng.normal(0.0, 1.0, (Hkv, T, nb))
    if case == "clustered_ties":
        S = np.round(S * 8.0) / 8.0
    elif case == "iid":
        S = rng.normal(0.0, 1.0, (Hkv, T, nb))
    elif case == "all_equal":
        S = np.full((Hkv, T, nb), 0.5)
    S32 = np.ascontiguousarray(S, np.float32)
    rows = np.arange(T)
    ref_sel = oracle.select(S32, B, off, rows, Ks)
    ref_u = oracle.union(ref_sel, W, nb)
    sel = torch.empty(Hkv, T, Ks, dtype=torch.int32, device="cuda")
    uo, ul, ub, um = s.alloc_union(p)
    st = s.new_status()
    s.sgqa_topk_union(p, torch.from_numpy(S32).cuda(), 0, T, sel, uo, ul, ub, um, status=st)
    assert s.read_status(st)[0] == 0
    assert np.array_equal(sel.cpu().numpy(), ref_sel)
    assert _gpu_union_lists(s, p, uo, ul, ub, um) == _oracle_union_lists(*ref_u)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("mode", [0, 1])
def test_sparse_attn_given_lists(s, name, mode):
    """R3: attention on the oracle's own block lists."""
    wl, inp = SMALL[name], inputs(name)
    p = s.params_for(wl, union_mode=mode)
    rows = np.arange(wl.seq_q)
    Q, K, V = widened(inp)
    S = oracle.scores(oracle.index_query(Q, wl.n_kv_heads, rows), oracle.merge_f64(K, wl.block_size),
                      wl.block_size, wl.q_offset, rows)
    sel = oracle.select(S, wl.block_size, wl.q_offset, rows, wl.k_blocks)
    uoff, ublk, umask = oracle.union(sel, wl.tile_q, wl.n_blocks)
    O64, lse64 = oracle.sparse_attn(Q, K, V, wl.q_offset, wl.block_size, sel, mode,
                                    (uoff, ublk, umask), wl.tile_q)
    d = dev_inputs(inp)
    O, lse = s.alloc_outputs(p)
    ws = s.alloc_workspace(p, s.WS_SPARSE_ATTN)
    st = s.new_status()
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], *_upload_union(uoff, ublk, umask,
                                                                    wl.n_kv_heads, 0),
                           O, lse, page_table=d["page_table"], ws=ws, status=st)
    assert s.read_status(st)[0] == 0
    r3_check(O.float().cpu().numpy(), lse.cpu().numpy(), O64, lse64,
             lse_tol=lse_tol_for(wl, inp, rows))


def test_sparse_attn_jump_in_second_half(s):
    """A stage whose first 64 keys pass the one-pass check against the row's
    reference maximum (15.5 above it in log2 units, within the 2^16 lazy
    margin) while one of its last 64 keys exceeds it by 16.5: the maximum is
    raised in place, O and the P already written for the first 64 keys are
    rescaled, and those keys keep their weight (half the needle's each).  Keys
    are exact multiples of one direction: every other selected key has the
    logit L0 of the row's first stage (about 5).  The needle sits in the second
    half of softmax group 0's second stage (union blocks 40-47 of stage 32-47),
    the raised keys in its first half (blocks 32-39)."""
    T, off, H, d, B = 16, 4096, 8, 128, 8
    wl = BASE.replace(name="jump", seq_q=T, seq_kv=off + T, q_offset=off, n_q_heads=H,
                      n_kv_heads=1, head_dim=d, block_size=B, topk_tokens=64 * B, tile_q=16)
    a = b = 6.25  # logit of a selected key: a * b / sqrt(d) * log2(e) = 4.98
    b_hi = 25.75  # blocks 32-39: 20.52, above L0 by 15.54
    c = 27.0      # the needle: 21.52, above L0 by 16.54
    Tkv = off + T
    Qf = np.zeros((T, H, d), np.float32)
    Qf[:, :, 0] = a
    Kf = np.zeros((Tkv, 1, d), np.float32)
    Kf[:, 0, 0] = -b                     # blocks 64 .. : never selected
    Kf[: 64 * B, 0, 0] = b               # blocks 0 .. 63: the selection of every query
    Kf[32 * B: 40 * B, 0, 0] = b_hi
    Kf[44 * B + 3, 0, 0] = c
    Vf = np.random.default_rng(7).normal(0.0, 1.0, (Tkv, 1, d)).astype(np.float32)
    inp = {"workload": wl, "Q": synth.to_bf16_bits(Qf), "K": synth.to_bf16_bits(Kf),
           "V": synth.to_bf16_bits(Vf)}
    p = s.params_for(wl)
    rows = np.arange(T)
    Q, K, V = widened(inp)
    S = oracle.scores(oracle.index_query(Q, 1, rows), oracle.merge_f64(K, B), B, off, rows)
    sel = oracle.select(S, B, off, rows, 64)
    assert (sel[0][:, :64] == np.arange(64)).all()  # the construction holds
    uoff, ublk, umask = oracle.union(sel, wl.tile_q, wl.n_blocks)
    O64, lse64 = oracle.sparse_attn(Q, K, V, off, B, sel, 0, (uoff, ublk, umask), wl.tile_q)
    d_ = dev_inputs(inp)
    O, lse = s.alloc_outputs(p)
    ws = s.alloc_workspace(p, s.WS_SPARSE_ATTN)
    st = s.new_status()
    s.sgqa_sparse_attn_fwd(p, d_["Q"], d_["K"], d_["V"], *_upload_union(uoff, ublk, umask, 1, 0),
                           O, lse, page_table=None, ws=ws, status=st)
    assert s.read_status(st)[0] == 0
    r3_check(O.float().cpu().numpy(), lse.cpu().numpy(), O64, lse64)
