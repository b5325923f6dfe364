"""Host-side logic of bench.py: the multi-rank reductions (gloo, two ranks on
the CPU) and the closed-form algorithmic work against a brute-force count."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench
import oracle
from block_sparse_long_sgqa_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    out[rank] = (bench.reduce_max(1.5 + rank), bench.reduce_sum(10 * (rank + 1)))
    bench.barrier()
    dist.destroy_process_group()


def test_reductions_two_ranks_gloo():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: (2.5, 30.0), 1: (2.5, 30.0)}


def test_reductions_single_process_identity():
    assert bench.reduce_max(3.25) == 3.25 and bench.reduce_sum(4.0) == 4.0


def test_algorithmic_matches_brute_force():
    wl = synth.WORKLOADS["gqa_32k"].replace(seq_q=300, seq_kv=420, q_offset=120, topk_tokens=128,
                                            n_q_heads=8, n_kv_heads=2)
    inp = synth.make_inputs(wl)
    Q, K, _ = (synth.widen(inp[x]) for x in "QKV")
    rows = np.arange(wl.seq_q, dtype=np.int32)
    S = oracle.scores(oracle.index_query(Q, 2, rows), oracle.merge_f64(K, 8), 8, wl.q_offset, rows)
    sel = oracle.select(S, 8, wl.q_offset, rows, wl.k_blocks)
    # attended keys: 8 per selected block plus the causal part of the current block
    keys = ((sel[0] >= 0).sum(1) * 8 + (wl.q_offset + rows) % 8 + 1).sum()
    alg = bench.algorithmic(wl, chunk=128)
    assert alg["attn_flops"] == wl.n_q_heads * keys * 4 * wl.head_dim
    assert alg["index_flops"] == np.isfinite(S).sum() * 2 * wl.head_dim
    assert abs(sum(alg["attn_flops_chunks"]) - alg["attn_flops"]) < 1e-6 * alg["attn_flops"]
    assert len(alg["attn_flops_chunks"]) == 3
