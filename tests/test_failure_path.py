"""The give-up path of a stalled pipeline wait, exercised without a fault.

Every pipeline wait in the kernels is bounded; when one runs out the kernel
raises a shared abort flag, every role stops at its next wait, the copies in
flight land, tensor memory is released, and SGQA_ERR_TIMEOUT goes to the
status buffer.  A debug request in word 3 of the status buffer makes the
first attention work item wait on a barrier that nothing arrives on (1 ms
limit), while its K and V loaders have copies in flight.  The test checks the
reported status, that the stream and context stay usable, and that the next
normal call on the same buffers matches the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import dev_inputs, r3_check, widened
from test_parity_steps import SMALL, _upload_union, inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["b8", "b4"])
def test_stalled_wait_reports_timeout_and_recovers(name):
    from block_sparse_long_sgqa_gb300 import sgqa as s

    wl, inp = SMALL[name], inputs(name)
    p = s.params_for(wl)
    rows = np.arange(wl.seq_q)
    Q, K, V = widened(inp)
    S = oracle.scores(oracle.index_query(Q, wl.n_kv_heads, rows), oracle.merge_f64(K, wl.block_size),
                      wl.block_size, wl.q_offset, rows)
    sel = oracle.select(S, wl.block_size, wl.q_offset, rows, wl.k_blocks)
    uoff, ublk, umask = oracle.union(sel, wl.tile_q, wl.n_blocks)
    O64, lse64 = oracle.sparse_attn(Q, K, V, wl.q_offset, wl.block_size, sel, 0,
                                    (uoff, ublk, umask), wl.tile_q)
    d = dev_inputs(inp)
    union = _upload_union(uoff, ublk, umask, wl.n_kv_heads, 0)
    O, lse = s.alloc_outputs(p)
    ws = s.alloc_workspace(p, s.WS_SPARSE_ATTN)
    st = s.new_status()
    st[3] = s.DEBUG_STALL
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], *union, O, lse,
                           page_table=d["page_table"], ws=ws, status=st)
    code, detail = s.read_status(st)
    assert code == s.ERR_TIMEOUT and detail == 220, (s.status_string(code), detail)
    assert int(st[2].item()) >= 1
    # the context and the stream are still usable
    x = torch.arange(1000, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 499500.0
    # the next call on the same buffers, with the request cleared, is correct
    s.reset_status(st)
    assert int(st[3].item()) == 0
    O.fill_(0)
    s.sgqa_sparse_attn_fwd(p, d["Q"], d["K"], d["V"], *union, O, lse,
                           page_table=d["page_table"], ws=ws, status=st)
    assert s.read_status(st)[0] == 0
    r3_check(O.float().cpu().numpy(), lse.cpu().numpy(), O64, lse64)
