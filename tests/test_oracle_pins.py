"""Pins for the CPU oracle: hand-derived fixtures, brute force, closed forms and
independent library routines.  Every test here runs without a GPU.

The steps follow "Inside Step 5 Preview" (StepFun blog), section "Sparse GQA":
block merge and the 8x indexer saving (paragraph "Reducing indexer's cost"),
top-k selection (paragraph "Trade-off between top-k and block size"), the
union of adjacent tokens' top-k (paragraph "Efficient implementation of sparse
attention") and the main path over selected plus current blocks (Figure 3).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


# --------------------------------------------------------------------------- merge

def test_merge_tree_order_fixture():
    g = gold("merge_tree_order.json")
    K = np.array(g["keys"], np.float32).reshape(8, 1, 1)
    kb = oracle.merge_tree_f32(K, g["B"])
    assert kb.shape == (1, 1, 1)
    assert kb[0, 0, 0] == np.float32(g["tree_f32"])
    assert oracle.merge_f64(K, g["B"])[0, 0, 0] == g["exact_mean"]


def test_merge_b1_is_identity():
    K = rnd(1, 37, 3, 16)
    assert np.array_equal(oracle.merge_tree_f32(K, 1), K.transpose(1, 0, 2))
    assert np.array_equal(oracle.merge_f64(K, 1), K.transpose(1, 0, 2).astype(np.float64))


def test_merge_constant_and_numpy_mean():
    K = np.repeat(rnd(2, 5, 2, 8), 8, axis=0)  # each block of 8 rows is constant
    kb = oracle.merge_tree_f32(K, 8)
    assert np.array_equal(kb, K[::8].transpose(1, 0, 2))
    K = rnd(3, 100, 2, 32)
    B = 4
    ref = K[: (100 // B) * B].astype(np.float64).reshape(-1, B, 2, 32).mean(axis=1).transpose(1, 0, 2)
    np.testing.assert_allclose(oracle.merge_f64(K, B), ref, rtol=0, atol=1e-15)
    # fp32 tree within a few ulp of the exact mean; the partial tail block is never merged
    kb = oracle.merge_tree_f32(K, B)
    assert kb.shape == (2, 25, 32)
    np.testing.assert_allclose(kb, ref, rtol=0, atol=4e-7 * np.abs(K).max())


def test_merge_block_range():
    K = rnd(4, 64, 1, 4)
    kb = oracle.merge_tree_f32(K, 8, 3, 6)
    assert np.isnan(kb[:, :3]).all() and np.isnan(kb[:, 6:]).all()
    assert np.array_equal(kb[:, 3:6], oracle.merge_tree_f32(K, 8)[:, 3:6])


# --------------------------------------------------------------------------- scores

def test_scores_fixture():
    g = gold("scores_small.json")
    K = np.array(g["K"], np.float32)[:, None, :]
    Q = np.array(g["Q"], np.float32)
    kb = oracle.merge_f64(K, g["B"])
    assert np.array_equal(kb, np.array(g["Kbar"], np.float64))
    rows = np.arange(Q.shape[0])
    qt = oracle.index_query(Q, g["Hkv"], rows)
    assert np.array_equal(qt, np.array(g["qt"], np.float64))
    S = oracle.scores(qt, kb, g["B"], g["q_offset"], rows)
    exp = np.array([[[-np.inf if v is None else v for v in r] for r in gg] for gg in g["scores"]])
    assert np.array_equal(S, exp)
    sel = oracle.select(S, g["B"], g["q_offset"], rows, 1)
    assert np.array_equal(sel, np.array(g["sel_k1"]))


def test_scores_vs_torch_einsum():
    T, H, Hkv, d, B, off = 50, 8, 2, 16, 4, 30
    Q, K = rnd(5, T, H, d), rnd(6, off + T, Hkv, d)
    rows = np.arange(T)
    S = oracle.scores(oracle.index_query(Q, Hkv, rows), oracle.merge_f64(K, B), B, off, rows)
    q = torch.from_numpy(Q).double().view(T, Hkv, H // Hkv, d).mean(2)
    kb = torch.from_numpy(K).double()[: (off + T) // B * B].view(-1, B, Hkv, d).mean(1)
    ref = torch.einsum("tgi,jgi->gtj", q, kb).numpy()
    nh = (off + rows) // B
    finite = np.arange(S.shape[2])[None, :] < nh[:, None]
    assert np.array_equal(np.isfinite(S[0]), finite)
    np.testing.assert_allclose(S[:, finite], ref[:, finite], rtol=1e-12, atol=1e-12)


def test_indexer_pair_count_8x():
    """The pages: block size 8 cuts indexer and top-k cost by 8x.  The number of
    scored (query, block) pairs falls by sum pos / sum floor(pos/8) -> 8."""
    T, d = 4096, 2
    K = rnd(7, T, 1, d)
    Q = rnd(8, T, 1, d)
    rows = np.arange(T)
    qt = oracle.index_query(Q, 1, rows)
    n1 = np.isfinite(oracle.scores(qt, oracle.merge_f64(K, 1), 1, 0, rows)).sum()
    n8 = np.isfinite(oracle.scores(qt, oracle.merge_f64(K, 8), 8, 0, rows)).sum()
    assert n1 == T * (T - 1) // 2
    ratio = n1 / n8
    assert 7.9 < ratio < 8.1
    assert abs(ratio - 8.0137) < 1e-3


# --------------------------------------------------------------------------- top-k

def test_select_ties_fixture():
    g = gold("select_ties.json")
    vals = [float(v) if v != "pad" else 99.0 for v in g["scores"]]
    S = np.array([[vals]], np.float32)
    for k, exp in g["expected"].items():
        sel = oracle.select(S, g["B"], g["q_offset"], np.array([0]), int(k))
        assert sel[0, 0].tolist() == exp, k
    # the same ranking holds for fp64 scores
    sel = oracle.select(S.astype(np.float64), g["B"], g["q_offset"], np.array([0]), 5)
    assert sel[0, 0].tolist() == g["expected"]["5"]


@pytest.mark.parametrize("seed", range(6))
def test_select_vs_stable_argsort(seed):
    rng = np.random.default_rng(seed)
    Hkv, n, nblk, B, off = 2, 40, 70, 2, 3
    rows = np.sort(rng.choice(100, n, replace=False)).astype(np.int32)
    S = rng.integers(-4, 5, (Hkv, n, nblk)).astype(np.float32)  # many ties
    if seed % 2:
        S = rng.standard_normal((Hkv, n, nblk)).astype(np.float32)
    for Ks in (1, 5, 17, 64):
        sel = oracle.select(S, B, off, rows, Ks)
        for g in range(Hkv):
            for r, t in enumerate(rows):
                nh = min((off + t) // B, nblk)
                order = np.argsort(-S[g, r, :nh].astype(np.float64), kind="stable")
                exp = sorted(order[:Ks].tolist())
                exp += [-1] * (Ks - len(exp))
                assert sel[g, r].tolist() == exp


def test_b1_is_per_token_topk():
    """With B = 1 the block keys are the keys themselves, so the selection is the
    per-token top-k of the group query against every earlier key."""
    T, H, Hkv, d = 64, 4, 2, 8
    Q, K = rnd(9, T, H, d), rnd(10, T, Hkv, d)
    rows = np.arange(T)
    qt = oracle.index_query(Q, Hkv, rows)
    S = oracle.scores(qt, oracle.merge_f64(K, 1), 1, 0, rows)
    sel = oracle.select(S, 1, 0, rows, 5)
    q = Q.astype(np.float64).reshape(T, Hkv, H // Hkv, d).mean(2)
    for g in range(Hkv):
        for t in range(T):
            s = K[:t, g].astype(np.float64) @ q[t, g]
            exp = sorted(np.argsort(-s, kind="stable")[:5].tolist())
            got = [x for x in sel[g, t].tolist() if x >= 0]
            assert got == exp


# --------------------------------------------------------------------------- union

def test_union_fixture():
    g = gold("union_small.json")
    uoff, ublk, umask = oracle.union(np.array(g["sel"], np.int32), g["W"], g["nblk"])
    assert uoff.tolist() == g["uoff"]
    assert ublk.tolist() == g["ublk"]
    assert umask.tolist() == g["umask"]


def test_union_set_algebra():
    rng = np.random.default_rng(11)
    Hkv, T, Ks, W, nblk = 3, 100, 6, 16, 40
    sel = np.full((Hkv, T, Ks), -1, np.int32)
    for g in range(Hkv):
        for t in range(T):
            n = rng.integers(0, Ks + 1)
            sel[g, t, :n] = np.sort(rng.choice(nblk, n, replace=False))
    uoff, ublk, umask = oracle.union(sel, W, nblk)
    ntiles = (T + W - 1) // W
    for g in range(Hkv):
        for tau in range(ntiles):
            a, b = uoff[g, tau], uoff[g, tau + 1]
            U = ublk[a:b].tolist()
            members = range(tau * W, min(T, tau * W + W))
            exp = sorted(set().union(*[set(x for x in sel[g, t] if x >= 0) for t in members]))
            assert U == exp
            for u, m in zip(U, umask[a:b].tolist()):
                for i, t in enumerate(members):
                    assert bool((m >> i) & 1) == (u in sel[g, t])
                assert m >> len(members) == 0


# --------------------------------------------------------------------------- attention

def _sdpa_ref(Q, K, V, off, allowed=None):
    """Dense causal GQA attention from torch (fp64, CPU), via an explicit mask."""
    T, H, d = Q.shape
    Tkv, Hkv, _ = K.shape
    G = H // Hkv
    q = torch.from_numpy(Q).double().permute(1, 0, 2)
    k = torch.from_numpy(K).double().permute(1, 0, 2).repeat_interleave(G, 0)
    v = torch.from_numpy(V).double().permute(1, 0, 2).repeat_interleave(G, 0)
    pos = off + torch.arange(T)
    mask = torch.arange(Tkv)[None, :] <= pos[:, None]
    if allowed is not None:
        mask = torch.from_numpy(allowed)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask)
    s = (q @ k.transpose(1, 2)) / math.sqrt(d)
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, -1)
    return o.permute(1, 0, 2).numpy(), lse.numpy()


def test_attn_fixture_two_keys():
    g = gold("attn_two_keys.json")
    Q, K, V = (np.array(g[x], np.float32) for x in ("Q", "K", "V"))
    O, lse = oracle.sparse_attn(Q, K, V, g["q_offset"], g["B"], np.array(g["sel"], np.int32),
                                scale=g["scale"])
    assert abs(O[0, 0, 0] - g["O"]) < 1e-6 and abs(lse[0, 0] - g["lse"]) < 1e-6
    O, lse = oracle.sparse_attn(Q, K, V, g["q_offset"], g["B"], np.full((1, 1, 1), -1, np.int32),
                                scale=g["scale"])
    assert O[0, 0, 0] == g["O_nosel"] and abs(lse[0, 0] - g["lse_nosel"]) < 1e-6


def test_attn_nothing_selected_b1_closed_form():
    """k = 0 and B = 1: only the query's own position is visible, so O = V[pos]
    and lse = scale * q . k_pos."""
    T, H, Hkv, d, off = 20, 4, 2, 8, 5
    Q, K, V = rnd(12, T, H, d), rnd(13, off + T, Hkv, d), rnd(14, off + T, Hkv, d)
    O, lse = oracle.sparse_attn(Q, K, V, off, 1, np.full((Hkv, T, 1), -1, np.int32))
    for t in range(T):
        for h in range(H):
            g = h // 2
            assert np.array_equal(O[t, h], V[off + t, g].astype(np.float64))
            exp = float(Q[t, h].astype(np.float64) @ K[off + t, g].astype(np.float64)) / math.sqrt(d)
            assert abs(lse[h, t] - exp) < 1e-12


@pytest.mark.parametrize("B,off", [(8, 0), (4, 13), (1, 7)])
def test_full_selection_is_dense_causal(B, off):
    """When k covers every historical block, block-sparse attention is dense
    causal GQA attention."""
    T, H, Hkv, d = 40, 4, 2, 16
    Q, K, V = rnd(15, T, H, d), rnd(16, off + T, Hkv, d), rnd(17, off + T, Hkv, d)
    rows = np.arange(T)
    nblk = (off + T) // B
    S, sel, O, lse = oracle.prefill_rows(Q, K, V, off, B, nblk, rows)
    Od, lsed = oracle.dense_attn(Q, K, V, off)
    Or, lser = _sdpa_ref(Q, K, V, off)
    np.testing.assert_allclose(O, Or, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lser, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Od, Or, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lsed, lser, rtol=0, atol=1e-12)


def test_sparse_attention_vs_masked_sdpa():
    """The mode-A key set: the selected blocks plus the causal part of the
    current block, checked against torch SDPA with that mask written out."""
    T, H, Hkv, d, B, off, Ks = 48, 4, 2, 16, 4, 20, 3
    Q, K, V = rnd(18, T, H, d), rnd(19, off + T, Hkv, d), rnd(20, off + T, Hkv, d)
    rows = np.arange(T)
    S, sel, O, lse = oracle.prefill_rows(Q, K, V, off, B, Ks, rows)
    G = H // Hkv
    allowed = np.zeros((H, T, off + T), bool)
    for h in range(H):
        for t in range(T):
            pos = off + t
            for j in sel[h // G, t]:
                if j >= 0:
                    allowed[h, t, j * B:(j + 1) * B] = True
            allowed[h, t, (pos // B) * B:pos + 1] = True
    Or, lser = _sdpa_ref(Q, K, V, off, allowed)
    np.testing.assert_allclose(O, Or, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lser, rtol=0, atol=1e-12)


def test_mode_b_contains_mode_a_and_w1_equal():
    T, H, Hkv, d, B, off, Ks = 40, 4, 2, 8, 2, 9, 3
    Q, K, V = rnd(21, T, H, d), rnd(22, off + T, Hkv, d), rnd(23, off + T, Hkv, d)
    rows = np.arange(T)
    _, sel, OA, lseA = oracle.prefill_rows(Q, K, V, off, B, Ks, rows)
    OB1, lseB1 = oracle.sparse_attn(Q, K, V, off, B, sel, mode=1, W=1)
    np.testing.assert_allclose(OB1, OA, rtol=0, atol=1e-13)
    OB, lseB = oracle.sparse_attn(Q, K, V, off, B, sel, mode=1, W=8)
    assert (lseB >= lseA - 1e-12).all()
    assert (lseB > lseA + 1e-9).any()


@pytest.mark.parametrize("B,W,off", [(2, 8, 5), (4, 16, 0), (1, 4, 3)])
def test_mode_b_allowed_set_vs_masked_sdpa(B, W, off):
    """Mode B's key set, written out by hand: every block of the query's tile
    union that lies strictly before the query's own block, plus the causal
    part of that block.  The selections are built so that later tile-mates
    select the earlier queries' current block and blocks past it (which mode B
    must hide from them), so dropping the cut or letting the current block in
    as a historical one changes the result."""
    T, H, Hkv, d, Ks = 48, 4, 2, 16, 3
    Q, K, V = rnd(31 + B, T, H, d), rnd(32 + B, off + T, Hkv, d), rnd(33 + B, off + T, Hkv, d)
    rng = np.random.default_rng(34 + B)
    sel = np.full((Hkv, T, Ks), -1, np.int32)
    for g in range(Hkv):
        for t in range(T):
            nh = (off + t) // B
            if nh == 0:
                continue
            # the most recent historical block, plus a few older ones
            older = rng.choice(nh - 1, size=min(Ks - 1, nh - 1), replace=False) if nh > 1 else []
            sel[g, t, :len(older) + 1] = sorted(list(older) + [nh - 1])
    # the hand-built allowed mask of mode B
    G = H // Hkv
    allowed = np.zeros((H, T, off + T), bool)
    n_cur = n_future = 0
    for g in range(Hkv):
        for t in range(T):
            tau = t // W
            mates = range(tau * W, min(tau * W + W, T))
            union = {int(j) for m in mates for j in sel[g, m] if j >= 0}
            cur = (off + t) // B
            n_cur += cur in union
            n_future += any(j > cur for j in union)
            for h in range(g * G, (g + 1) * G):
                for j in union:
                    if j < cur:
                        allowed[h, t, j * B:(j + 1) * B] = True
                allowed[h, t, cur * B:off + t + 1] = True
    assert n_cur > 0 and n_future > 0  # both branches of the cut are exercised
    O, lse = oracle.sparse_attn(Q, K, V, off, B, sel, mode=1, W=W)
    Or, lser = _sdpa_ref(Q, K, V, off, allowed)
    np.testing.assert_allclose(O, Or, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lser, rtol=0, atol=1e-12)


def test_coverage_monotone_in_k():
    """Selections are nested in k (one total order), so the attention mass they
    cover, exp(lse_sparse - lse_dense), never decreases with k and reaches 1."""
    T, H, Hkv, d, B = 64, 4, 1, 16, 4
    Q, K, V = rnd(24, T, H, d), rnd(25, T, Hkv, d), rnd(26, T, Hkv, d)
    rows = np.arange(T)
    _, lsed = oracle.dense_attn(Q, K, V, 0)
    prev = None
    for Ks in (1, 2, 4, 8, 16):
        _, sel, _, lse = oracle.prefill_rows(Q, K, V, 0, B, Ks, rows)
        cov = np.exp(lse - lsed)
        assert (cov <= 1 + 1e-12).all()
        if prev is not None:
            assert (cov >= prev - 1e-12).all()
        prev = cov
    assert np.allclose(prev, 1.0, atol=1e-12)


# --------------------------------------------------------------------------- inputs

def test_synth_is_seeded_and_normal():
    a = synth.normal(5, 1, 100000)
    assert np.array_equal(a, synth.normal(5, 1, 100000))
    assert not np.array_equal(a, synth.normal(6, 1, 100000))
    assert abs(a.mean()) < 0.02 and abs(a.std() - 1) < 0.02


def test_synth_bf16_rounding():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e38], np.float32)
    b = synth.to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(b)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(back, ref)


def test_synth_workload_small():
    wl = synth.WORKLOADS["gqa_32k"].replace(seq_q=256, seq_kv=256)
    inp = synth.make_inputs(wl)
    assert inp["Q"].shape == (256, 32, 128) and inp["Q"].dtype == np.uint16
    assert inp["K"].shape == (256, 4, 128)
    q = synth.widen(inp["Q"])
    # AR(1) query noise: neighbours correlate, marginals stay ~N(0,1)
    assert 0.8 < q.std() < 1.3
    wl = synth.WORKLOADS["step5_128k"].replace(seq_q=512, seq_kv=512)
    inp = synth.make_inputs(wl)
    assert inp["needles"].shape == (8, 8, 16)


# ------------------------------------------------------ attention backward (training side)

def _grid(seed, *shape):
    """Values on a 2^-6 grid in [-1, 1]: x +- 2^-10 is exact in fp32."""
    return (np.random.default_rng(seed).integers(-64, 65, shape) / 64.0).astype(np.float32)


def _rand_sel(seed, Hkv, T, off, B, Ks):
    """A valid selection: per (group, query) min(Ks, nh) distinct historical
    blocks, ascending, -1 padded."""
    rng = np.random.default_rng(seed)
    sel = np.full((Hkv, T, Ks), -1, np.int32)
    for g in range(Hkv):
        for t in range(T):
            nh = (off + t) // B
            k = min(Ks, nh)
            if k:
                sel[g, t, :k] = np.sort(rng.choice(nh, size=k, replace=False))
    return sel


@pytest.mark.parametrize("mode", [0, 1])
def test_attn_bwd_finite_differences(mode):
    """The attention backward against central differences of L = sum(dO * O)
    through the forward oracle, on entries of Q, K and V (modes A and B)."""
    T, H, Hkv, d, B, off, Ks, W = 6, 4, 2, 8, 2, 6, 2, 4
    Q, K, V = _grid(30, T, H, d), _grid(31, off + T, Hkv, d), _grid(32, off + T, Hkv, d)
    sel = _rand_sel(33, Hkv, T, off, B, Ks)
    dO = np.random.default_rng(34).standard_normal((T, H, d))
    dQ, dK, dV = oracle.sparse_attn_bwd(Q, K, V, dO, off, B, sel, mode=mode, W=W)

    def loss(X, which):
        args = {"Q": (X, K, V), "K": (Q, X, V), "V": (Q, K, X)}[which]
        O, _ = oracle.sparse_attn(*args, off, B, sel, mode=mode, W=W)
        return float((dO * O).sum())

    eps = 2.0 ** -10
    rng = np.random.default_rng(35)
    for which, X, grad in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        for _ in range(8):
            idx = tuple(int(rng.integers(0, n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            fd = (loss(Xp, which) - loss(Xm, which)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 + 1e-6 * abs(fd), (which, idx, fd, grad[idx])


def test_attn_bwd_full_selection_vs_autograd():
    """With every historical block selected, the backward is that of dense
    causal GQA attention: torch autograd in fp64."""
    T, H, Hkv, d, B, off = 20, 4, 2, 8, 4, 12
    Q, K, V = rnd(36, T, H, d), rnd(37, off + T, Hkv, d), rnd(38, off + T, Hkv, d)
    nblk = (off + T) // B
    sel = np.full((Hkv, T, nblk), -1, np.int32)
    for t in range(T):
        nh = (off + t) // B
        sel[:, t, :nh] = np.arange(nh)
    dO = np.random.default_rng(39).standard_normal((T, H, d))
    dQ, dK, dV = oracle.sparse_attn_bwd(Q, K, V, dO, off, B, sel)
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    G, scale = H // Hkv, 1.0 / math.sqrt(d)
    pos = off + torch.arange(T)
    allowed = torch.arange(off + T)[None, :] <= pos[:, None]
    outs = []
    for h in range(H):
        s = scale * q[:, h] @ k[:, h // G].T
        outs.append(torch.softmax(s.masked_fill(~allowed, float("-inf")), -1) @ v[:, h // G])
    (torch.stack(outs, 1) * torch.tensor(dO)).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=0, atol=1e-11)


def test_attn_bwd_invariants():
    """Each row's weights sum to one and its score gradients to zero: the sum
    of dV over a group's keys is the sum of dO over the group's query heads,
    the sum of dK over them is zero, and dQ does not change when one vector is
    added to every key."""
    T, H, Hkv, d, B, off, Ks = 16, 4, 2, 8, 2, 10, 3
    Q, K, V = _grid(40, T, H, d), _grid(41, off + T, Hkv, d), _grid(42, off + T, Hkv, d)
    sel = _rand_sel(43, Hkv, T, off, B, Ks)
    dO = np.random.default_rng(44).standard_normal((T, H, d))
    dQ, dK, dV = oracle.sparse_attn_bwd(Q, K, V, dO, off, B, sel)
    G = H // Hkv
    for g in range(Hkv):
        np.testing.assert_allclose(dV[:, g].sum(0), dO[:, g * G:(g + 1) * G].sum((0, 1)),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(dK[:, g].sum(0), 0.0, rtol=0, atol=1e-12)
    c = _grid(45, d)
    dQ2, _, _ = oracle.sparse_attn_bwd(Q, K + c[None, None, :], V, dO, off, B, sel)
    np.testing.assert_allclose(dQ2, dQ, rtol=0, atol=1e-11)


# --------------------------------------------------------------------------- bf16 indexer

def _bf16_case_scores(q, k):
    q = np.array(q, np.float32)[None, None, :]          # [1 row][1 group][d]
    k = np.array(k, np.float32)[None, None, :]          # [1 group][1 block][d]
    return oracle.scores_bf16(q, k, 1, 1, np.array([0], np.int32))[0, 0, 0]


def test_scores_bf16_fixture():
    """Hand-worked sums and tie cases of the bf16 indexer (tests/golden/scores_bf16.json)."""
    for c in gold("scores_bf16.json")["cases"]:
        assert _bf16_case_scores(c["q"], c["k"]) == np.float32(c["score"]), c


def test_scores_bf16_operand_rounding_vs_torch():
    """Against a unit key the score is the query element rounded to bf16:
    compare with torch's own fp32 -> bfloat16 conversion."""
    q = rnd(40, 64).astype(np.float32) * np.float32(37.0)
    ref = torch.from_numpy(q).to(torch.bfloat16).float().numpy()
    for i in range(64):
        e = np.zeros(64, np.float32)
        e[i] = 1.0
        assert _bf16_case_scores(q, e) == ref[i], i


def test_scores_bf16_integer_sums_vs_torch():
    """Integer operands make every sum exact in fp32, so torch's fp32 ->
    bfloat16 rounding of the exact dot product is the reference; also the
    causal -inf pattern."""
    rng = np.random.default_rng(41)
    Hkv, nblk, d, B, off = 2, 40, 128, 4, 37
    qt = rng.integers(-20, 21, size=(5, Hkv, d)).astype(np.float32)
    kb = rng.integers(-20, 21, size=(Hkv, nblk, d)).astype(np.float32)
    rows = np.array([0, 3, 50, 90, 120], np.int32)
    S = oracle.scores_bf16(qt, kb, B, off, rows)
    exact = np.einsum("rgi,gji->grj", qt.astype(np.float64), kb.astype(np.float64))
    ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).float().numpy()
    nh = (off + rows) // B
    for r in range(len(rows)):
        n = min(nh[r], nblk)
        assert np.array_equal(S[:, r, :n], ref[:, r, :n])
        assert (S[:, r, n:] == -np.inf).all()
    assert (np.abs(exact) > 512).any()  # sums large enough for the rounding to drop bits
