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
from helpers import dev_inputs
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
