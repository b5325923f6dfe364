"""The indexer's variants against the oracle, through the C ABI.

* The bf16 indexer (SGQA_INDEX_BF16): one bf16 product per score, each score
  rounded to bf16.  Scores against the oracle's bf16 definition (within one
  bf16 unit in the last place: the tensor cores sum in fp32, the oracle
  exactly); selections exact on the GPU's own scores (R1) and the fused call
  equal to the step composition bit for bit; recall of the exact (split)
  selection reported and bounded below.
* Separate index inputs (sgqa_prefill_ex): index queries [T][Hkv][d] and index
  keys in K's layout, end to end against the oracle; with none given the call
  equals sgqa_prefill bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth
from helpers import clear_margin, dev_inputs, r2_check, r3_check, to_dev, widened
from test_parity_steps import SMALL, _gpu_union_lists, _oracle_union_lists, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s():
    from block_sparse_long_sgqa_gb300 import sgqa

    return sgqa


FILT = synth.WORKLOADS["gqa_32k"].replace(name="filt", seq_q=2048, seq_kv=22528, q_offset=20480)


def _gpu_scores(s, p, Q, Kbar, q0, q1):
    sc = torch.empty(p.n_kv_heads, q1 - q0, p.seq_kv // p.block_size, device="cuda")
    s.sgqa_index_scores(p, Q, Kbar, q0, q1, sc, s.alloc_workspace(p, s.WS_INDEX_SCORES))
    return sc


@pytest.mark.parametrize("name", ["b8", "b16", "d64_g2", "paged"])
def test_index_scores_bf16_vs_oracle(s, name):
    wl, inp = SMALL[name], inputs(name)
    p = s.params_for(wl, index_mode=s.INDEX_BF16)
    d = dev_inputs(inp)
    Q, K, _ = widened(inp)
    Kbar = s.kbar_empty(p)
    s.sgqa_block_merge(p, d["K"], Kbar, page_table=d["page_table"])
    rows = np.arange(wl.seq_q, dtype=np.int32)
    got = _gpu_scores(s, p, d["Q"], Kbar, 0, wl.seq_q).cpu().numpy()
    qt32 = oracle.index_query(Q, wl.n_kv_heads, rows).astype(np.float32)
    kb32 = oracle.merge_tree_f32(K, wl.block_size)
    ref = oracle.scores_bf16(qt32, kb32, wl.block_size, wl.q_offset, rows)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin) and (got[~fin] == -np.inf).all()
    # every GPU score is a bf16 value
    assert (got[fin].view(np.uint32) & 0xFFFF == 0).all()
    # one bf16 ulp (<= 2^-7 |s|), plus an operand that rounded the other way
    prod = np.einsum("rgi,gji->grj", np.abs(qt32.astype(np.float64)), np.abs(kb32.astype(np.float64)))
    bound = 2.0 ** -7 * np.abs(ref.astype(np.float64)) + 2.0 ** -8 * prod + 1e-30
    err = np.abs(got[fin].astype(np.float64) - ref[fin])
    assert (err <= bound[fin]).all(), float((err / bound[fin]).max())
    assert (got[fin] == ref[fin]).mean() > 0.98


@pytest.mark.parametrize("case", ["b8", "filt"])
def test_prefill_bf16_index_equals_composition(s, case):
    """The fused prefill with the bf16 indexer equals the steps called one by
    one (bf16 scores -> top-k and union -> attention), bit for bit; "filt"
    selects from threshold candidates, where bf16 rounding makes exact ties
    frequent.  Selection and union also bit-exact against the oracle on the
    GPU's own bf16 scores (R1)."""
    wl = SMALL["b8"] if case == "b8" else FILT
    inp = inputs("b8") if case == "b8" else synth.make_inputs(wl)
    p = s.params_for(wl, index_mode=s.INDEX_BF16)
    d = dev_inputs(inp)
    O, lse = s.alloc_outputs(p)
    Kbar = s.kbar_empty(p)
    st = s.new_status()
    s.sgqa_prefill(p, d["Q"], d["K"], d["V"], Kbar, O, lse, s.alloc_workspace(p, s.WS_PREFILL),
                   page_table=d["page_table"], status=st)
    assert s.read_status(st)[0] == 0
    sc = _gpu_scores(s, p, d["Q"], Kbar, 0, wl.seq_q)
    sel = torch.empty(wl.n_kv_heads, wl.seq_q, wl.k_blocks, dtype=torch.int32, device="cuda")
    u = s.alloc_union(p)
    s.sgqa_topk_union(p, sc, 0, wl.seq_q, sel, *u, status=st)
    O2, l2 = s.alloc_outputs(p)
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], *u, O2, l2, page_table=d["page_table"],
                           ws=s.alloc_workspace(p, s.WS_SPARSE_ATTN), status=st)
    assert s.read_status(st)[0] == 0
    assert torch.equal(O, O2) and torch.equal(lse, l2)
    S32 = sc.cpu().numpy()
    rows = np.arange(wl.seq_q, dtype=np.int32)
    ref_sel = oracle.select(S32, wl.block_size, wl.q_offset, rows, wl.k_blocks)
    assert np.array_equal(sel.cpu().numpy(), ref_sel)
    assert _gpu_union_lists(s, p, *u) == _oracle_union_lists(*oracle.union(ref_sel, wl.tile_q,
                                                                           wl.n_blocks))


def test_bf16_index_recall_of_exact_selection(s):
    """Recall of the exact (split-indexer) selection by the bf16 indexer's, on
    the clustered 32K shape's last 512 queries (rows of 3.5-4K blocks, 256
    selected), and the bf16 selection checked against the oracle's bf16
    scores: where it differs, both scores lie within two bf16 ulps of the
    k-th."""
    wl = synth.WORKLOADS["gqa_32k"].replace(name="rec", seq_q=512, q_offset=32768 - 512)
    inp = synth.make_inputs(wl)
    d = dev_inputs(inp)
    sels = {}
    for mode in (s.INDEX_SPLIT, s.INDEX_BF16):
        p = s.params_for(wl, index_mode=mode)
        Kbar = s.kbar_empty(p)
        s.sgqa_block_merge(p, d["K"], Kbar)
        sc = _gpu_scores(s, p, d["Q"], Kbar, 0, wl.seq_q)
        sel = torch.empty(wl.n_kv_heads, wl.seq_q, wl.k_blocks, dtype=torch.int32, device="cuda")
        u = s.alloc_union(p)
        s.sgqa_topk_union(p, sc, 0, wl.seq_q, sel, *u)
        sels[mode] = sel.cpu().numpy()
    a, b = sels[s.INDEX_SPLIT], sels[s.INDEX_BF16]
    hit = sum(len(np.intersect1d(a[g, r], b[g, r])) for g in range(a.shape[0]) for r in range(a.shape[1]))
    recall = hit / a.size
    assert recall > 0.9, recall
    # against the oracle's bf16 scores
    Q, K, _ = widened(inp)
    rows = np.arange(wl.seq_q, dtype=np.int32)
    qt32 = oracle.index_query(Q, wl.n_kv_heads, rows).astype(np.float32)
    Sb = oracle.scores_bf16(qt32, oracle.merge_tree_f32(K, 8), 8, wl.q_offset, rows).astype(np.float64)
    for g in range(b.shape[0]):
        for r in range(b.shape[1]):
            srt = np.sort(Sb[g, r][np.isfinite(Sb[g, r])])[::-1]
            sk = srt[wl.k_blocks - 1]
            ref = set(np.argsort(-Sb[g, r], kind="stable")[:wl.k_blocks].tolist())
            for j in ref.symmetric_difference(b[g, r].tolist()):
                assert abs(Sb[g, r, j] - sk) <= 2 * 2.0 ** -7 * abs(sk), (g, r, j)


@pytest.mark.parametrize("name", ["b8", "paged"])
def test_prefill_ex_index_inputs_vs_oracle(s, name):
    """Separate index queries and keys: the block keys are the index keys'
    block means, the group's index query is used as is, the attention still
    reads Q, K and V."""
    wl, inp = SMALL[name], inputs(name)
    rng = np.random.default_rng(5)
    Qi = rng.standard_normal((wl.seq_q, wl.n_kv_heads, wl.head_dim)).astype(np.float32) * 2.0
    Ki = rng.standard_normal((wl.seq_kv, wl.n_kv_heads, wl.head_dim)).astype(np.float32)
    Qi_b, Ki_b = synth.to_bf16_bits(Qi), synth.to_bf16_bits(Ki)
    d = dev_inputs(inp)
    dQi = to_dev(Qi_b)
    dKi = to_dev(synth.to_paged(Ki_b, inp["page_table"], wl.page_size) if wl.page_size else Ki_b)
    p = s.params_for(wl)
    O, lse = s.alloc_outputs(p)
    Kbar = s.kbar_empty(p)
    st = s.new_status()
    ws = s.alloc_workspace(p, s.WS_PREFILL)
    s.sgqa_prefill_ex(p, d["Q"], d["K"], d["V"], Kbar, O, lse, ws, Qidx=dQi, Kidx=dKi,
                      page_table=d["page_table"], status=st)
    assert s.read_status(st)[0] == 0
    Q, K, V = widened(inp)
    Qw, Kw = synth.widen(Qi_b), synth.widen(Ki_b)
    assert np.array_equal(Kbar.cpu().numpy().view(np.uint32),
                          oracle.merge_tree_f32(Kw, wl.block_size).view(np.uint32))
    rows = np.arange(wl.seq_q, dtype=np.int32)
    S, sel_rows, O64, lse64 = oracle.prefill_rows(Q, K, V, wl.q_offset, wl.block_size,
                                                  wl.k_blocks, rows, Qidx=Qw, Kidx=Kw)
    clear = clear_margin(S, wl, rows)
    G = wl.n_q_heads // wl.n_kv_heads
    mask = np.repeat(clear.T, G, axis=1)
    assert mask.mean() > 0.9
    r3_check(O.float().cpu().numpy(), lse.cpu().numpy(), O64, lse64, mask)
    # R2 on the standalone selection: scores of the index queries (one head per group)
    pi = s.params(wl.seq_q, wl.seq_kv, wl.q_offset, wl.n_kv_heads, wl.n_kv_heads, wl.head_dim,
                  wl.block_size, wl.topk_tokens, wl.tile_q, wl.page_size)
    sc = _gpu_scores(s, pi, dQi, Kbar, 0, wl.seq_q)
    sel = torch.empty(wl.n_kv_heads, wl.seq_q, wl.k_blocks, dtype=torch.int32, device="cuda")
    u = s.alloc_union(p)
    s.sgqa_topk_union(p, sc, 0, wl.seq_q, sel, *u, status=st)
    r2_check(sel.cpu().numpy(), S, wl, rows)
    # the composition equals the fused call bit for bit
    O2, l2 = s.alloc_outputs(p)
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], *u, O2, l2, page_table=d["page_table"],
                           ws=s.alloc_workspace(p, s.WS_SPARSE_ATTN), status=st)
    assert s.read_status(st)[0] == 0
    assert torch.equal(O, O2) and torch.equal(lse, l2)
    # with no index inputs, sgqa_prefill_ex is sgqa_prefill
    O3, l3 = s.alloc_outputs(p)
    Kb3 = s.kbar_empty(p)
    s.sgqa_prefill_ex(p, d["Q"], d["K"], d["V"], Kb3, O3, l3, ws, page_table=d["page_table"])
    O4, l4 = s.alloc_outputs(p)
    Kb4 = s.kbar_empty(p)
    s.sgqa_prefill(p, d["Q"], d["K"], d["V"], Kb4, O4, l4, ws, page_table=d["page_table"])
    assert torch.equal(O3, O4) and torch.equal(l3, l4) and torch.equal(Kb3, Kb4)
