"""Decode steps (sgqa_decode): one query at the end of a long paged cache,
with a persistent block-key cache and the attention split over ranges of its
selected blocks.

* A step against the oracle end to end (R3 on clear-margin rows, R2 on the
  standalone selection), at a position that selects from threshold
  candidates and one that takes the CTA-per-row select.
* A loop of steps crossing block boundaries with one cache: every step equals
  sgqa_prefill on the same params (same selection, so the same keys; the
  split attention is merged in a fixed order and rounds P to bf16 against
  its own running maxima, so O differs from the unsplit one by that rounding
  noise: within max-abs 2e-3 and mean-abs 2e-4, ten times tighter than R3,
  and lse within 1e-5),
  the cache's block keys end up bit-exact against the oracle's merge and its
  split halves consistent with them, and valid_blocks follows the steps.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_sgqa_gb300 import synth
from helpers import clear_margin, dev_inputs, lse_tol_for, r3_check, widened
from test_parity_prefill import check_end_to_end, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s():
    from block_sparse_long_sgqa_gb300 import sgqa

    return sgqa


def decode_wl(pos, Tkv=None):
    return synth.WORKLOADS["chunk_1m"].replace(name="decode", seq_q=1, q_offset=pos,
                                               seq_kv=pos + 1 if Tkv is None else Tkv)


@pytest.mark.parametrize("pos", [20000, 150001])
def test_decode_step_vs_oracle(s, pos):
    wl = decode_wl(pos)
    inp = synth.make_inputs(wl)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    cache = s.KeyCache(p, cap_blocks=(pos + 4096) // wl.block_size)
    O, lse = s.alloc_outputs(p)
    st = s.new_status()
    s.sgqa_decode(p, d["Q"], d["K"], d["V"], cache, O, lse, s.alloc_workspace(p, s.WS_DECODE),
                  page_table=d["page_table"], status=st)
    assert s.read_status(st)[0] == 0
    assert cache.valid_blocks == wl.n_blocks
    Kbar = cache.Kbar[:, :wl.n_blocks].contiguous()
    _, frac = check_end_to_end(s, wl, inp, O, lse, np.arange(1, dtype=np.int32), Kbar, d)
    assert frac >= 0.5


def test_decode_loop_persistent_cache(s):
    p0, steps = 20000 - 10, 20
    big = decode_wl(p0 + steps - 1)
    inp = synth.make_inputs(big.replace(seq_q=steps, q_offset=p0))  # the queries of every step
    d = dev_inputs(inp)
    cap = (p0 + steps + 4096) // big.block_size
    cache = None
    ws = None
    for i in range(steps):
        wl = decode_wl(p0 + i)
        p = s.params_for(wl)
        if cache is None:
            cache = s.KeyCache(p, cap_blocks=cap)
            ws = s.alloc_workspace(s.params_for(decode_wl(p0 + steps - 1)), s.WS_DECODE)
        assert s.workspace_bytes(p, s.WS_DECODE) <= ws.numel()
        Qi = d["Q"][i:i + 1].contiguous()
        O, lse = s.alloc_outputs(p)
        st = s.new_status()
        s.sgqa_decode(p, Qi, d["K"], d["V"], cache, O, lse, ws, page_table=d["page_table"],
                      status=st)
        assert s.read_status(st)[0] == 0
        assert cache.valid_blocks == wl.n_blocks
        O2, l2, _ = run_prefill(s, p, dict(d, Q=Qi))
        diff = (O.float() - O2.float()).abs()
        # the split and unsplit attention round P to bf16 against different
        # running maxima, so each carries its own rounding noise (measured
        # about 3e-4 of O against the fp64 oracle for either; 5e-4 apart)
        assert diff.max().item() <= 2e-3 and diff.mean().item() <= 2e-4, float(diff.max())
        assert (lse - l2).abs().max().item() <= 1e-5
    # the cache: every block merged once, bit-exact, and split into hi/lo halves
    nb = (p0 + steps) // big.block_size
    K = synth.widen(inp["K"])
    ref = oracle.merge_tree_f32(K, big.block_size)[:, :nb]
    assert np.array_equal(cache.Kbar[:, :nb].cpu().numpy().view(np.uint32), ref.view(np.uint32))
    hi = cache.Ksplit[0, :, :nb].float()
    lo = cache.Ksplit[1, :, :nb].float()
    assert torch.equal(hi, cache.Kbar[:, :nb].to(torch.bfloat16).float())
    assert (hi + lo - cache.Kbar[:, :nb]).abs().max().item() <= 2.0 ** -16 * cache.Kbar[:, :nb].abs().max().item()


@pytest.mark.parametrize("pos", [0, 5, 256, 300])
def test_decode_edge_positions(s, pos):
    """Decode steps at the edges of the selection, on small heads: the first
    position (no block before it), inside the first block, at the first
    position after exactly k/B blocks (all of them attended), and past it
    (a real selection); each step against the oracle, the cache's blocks
    bit-exact against the oracle's merge."""
    wl = synth.WORKLOADS["step5_128k"].replace(name="dec_edge", seq_q=1, q_offset=pos,
                                               seq_kv=pos + 1, n_q_heads=32, n_kv_heads=4,
                                               topk_tokens=256, needles=0)
    inp = synth.make_inputs(wl)
    p = s.params_for(wl)
    d = dev_inputs(inp)
    cache = s.KeyCache(p, cap_blocks=64)
    O, lse = s.alloc_outputs(p)
    st = s.new_status()
    s.sgqa_decode(p, d["Q"], d["K"], d["V"], cache, O, lse, s.alloc_workspace(p, s.WS_DECODE),
                  page_table=d["page_table"], status=st)
    assert s.read_status(st)[0] == 0
    nb = (pos + 1) // wl.block_size
    assert cache.valid_blocks == nb
    Q, K, V = widened(inp)
    rows = np.arange(1, dtype=np.int32)
    S, _, O64, lse64 = oracle.prefill_rows(Q, K, V, wl.q_offset, wl.block_size, wl.k_blocks, rows)
    G = wl.n_q_heads // wl.n_kv_heads
    mask = np.repeat(clear_margin(S, wl, rows).T, G, axis=1)
    assert mask.mean() >= 0.5
    r3_check(O.float().cpu().numpy(), lse.cpu().numpy(), O64, lse64, mask,
             lse_tol=lse_tol_for(wl, inp, rows))
    if nb:
        ref = oracle.merge_tree_f32(synth.widen(inp["K"]), wl.block_size)[:, :nb]
        assert np.array_equal(cache.Kbar[:, :nb].cpu().numpy().view(np.uint32), ref.view(np.uint32))
