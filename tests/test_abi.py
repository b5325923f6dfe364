"""Host-only checks of the C ABI: the library loads without a GPU, exports
every entry point include/sgqa.h declares, and rejects bad arguments on the
host before touching CUDA."""
import ctypes
import os
import re

import pytest

import oracle
from block_sparse_long_sgqa_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def s():
    from block_sparse_long_sgqa_gb300 import sgqa

    return sgqa


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "sgqa.h")).read()
    return sorted(set(re.findall(r"SGQA_API\s+[\w\s\*]+?\b(sgqa_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(s):
    decl = declared_symbols()
    assert len(decl) >= 11
    for name in decl:
        assert hasattr(s._lib, name), name
    assert set(decl) == set(s.EXPORTED)


def test_version_and_strings(s):
    assert s.version() == 100
    assert s.status_string(0) == "ok"
    for c in range(1, 9):
        assert s.status_string(c) not in ("ok", "unknown status")
    assert s.status_string(99) == "unknown status"


def p_small(s, **kw):
    base = dict(seq_q=300, seq_kv=300, q_offset=0, n_q_heads=8, n_kv_heads=2, head_dim=128,
                block_size=8, topk_tokens=64, tile_q=64)
    base.update(kw)
    return s.params(**base)


def test_workspace_and_capacity(s):
    p = p_small(s)
    for w in (s.WS_INDEX_SCORES, s.WS_TOPK_UNION, s.WS_PREFILL):
        assert s.workspace_bytes(p, w) > 0
    assert s.workspace_bytes(p, 99) == 0
    assert s.workspace_bytes(p_small(s, seq_q=0), s.WS_PREFILL) == 0
    # capacity: sum over groups and tiles of min(|tile| * k/B, nh(last query))
    T, W, B, Ks, Hkv = 300, 64, 8, 8, 2
    exp = 0
    for tau in range((T + W - 1) // W):
        n = min(W, T - tau * W)
        exp += min(n * Ks, (tau * W + n - 1) // B)
    assert s.union_capacity(p) == exp * Hkv
    assert s.union_capacity(p_small(s, n_q_heads=7)) == -1


def test_capacity_bounds_oracle_union(s):
    """The oracle's union of a random selection never exceeds the capacity."""
    import numpy as np

    wl = synth.WORKLOADS["gqa_32k"].replace(seq_q=200, seq_kv=200, n_q_heads=8, n_kv_heads=2,
                                            topk_tokens=32, tile_q=16)
    inp = synth.make_inputs(wl)
    Q, K, V = (synth.widen(inp[x]) for x in "QKV")
    rows = np.arange(wl.seq_q)
    S = oracle.scores(oracle.index_query(Q, 2, rows), oracle.merge_f64(K, 8), 8, 0, rows)
    sel = oracle.select(S, 8, 0, rows, 4)
    uoff, ublk, _ = oracle.union(sel, 16, wl.n_blocks)
    assert len(ublk) <= s.union_capacity(s.params_for(wl))


def _call_prefill(s, p, Q=0x1000, K=0x1000, V=0x1000, O=0x1000, lse=0x1000, Kbar=0x1000,
                  ws=0x1000, ws_bytes=1 << 40, pt=None, kvalid=0):
    vp = ctypes.c_void_p
    return s._lib.sgqa_prefill(ctypes.byref(p), vp(Q), vp(K), vp(V), vp(pt) if pt else None,
                               vp(Kbar), kvalid, vp(O), vp(lse), vp(ws), ws_bytes, None, None)


def test_host_validation_codes(s):
    assert _call_prefill(s, p_small(s, seq_q=0)) == s.ERR_INVALID_ARG
    assert _call_prefill(s, p_small(s, seq_kv=100)) == s.ERR_INVALID_ARG       # Tkv < off + T
    assert _call_prefill(s, p_small(s, n_q_heads=7)) == s.ERR_INVALID_ARG
    assert _call_prefill(s, p_small(s, topk_tokens=60)) == s.ERR_INVALID_ARG    # not a multiple of B
    assert _call_prefill(s, p_small(s, head_dim=96)) == s.ERR_UNSUPPORTED
    assert _call_prefill(s, p_small(s, block_size=3, topk_tokens=63)) == s.ERR_UNSUPPORTED
    assert _call_prefill(s, p_small(s, tile_q=65)) == s.ERR_UNSUPPORTED
    assert _call_prefill(s, p_small(s, page_size=12, seq_kv=300)) == s.ERR_UNSUPPORTED
    assert _call_prefill(s, p_small(s), Q=0) == s.ERR_INVALID_ARG               # null pointer
    assert _call_prefill(s, p_small(s), K=0x1008) == s.ERR_ALIGNMENT
    assert _call_prefill(s, p_small(s), ws_bytes=16) == s.ERR_WORKSPACE
    assert _call_prefill(s, p_small(s), kvalid=10**6) == s.ERR_INVALID_ARG
    # paged layout needs a page table, and a page table needs a paged layout
    assert _call_prefill(s, p_small(s, page_size=64, seq_kv=320)) == s.ERR_INVALID_ARG
    assert _call_prefill(s, p_small(s), pt=0x2000) == s.ERR_INVALID_ARG


def test_topk_union_range_validation(s):
    p = p_small(s)
    vp = ctypes.c_void_p
    f = s._lib.sgqa_topk_union
    args = lambda qb, qe, cap: (ctypes.byref(p), vp(0x1000), qb, qe, None, vp(0x1000), vp(0x1000),
                                vp(0x1000), vp(0x1000), cap, vp(0x1000), 1 << 40, None, None)
    assert f(*args(10, 64, 1 << 30)) == s.ERR_INVALID_ARG      # q_begin not tile aligned
    assert f(*args(0, 70, 1 << 30)) == s.ERR_INVALID_ARG       # q_end not tile aligned nor T
    assert f(*args(0, 301, 1 << 30)) == s.ERR_INVALID_ARG
    assert f(*args(0, 64, 1)) == s.ERR_WORKSPACE               # union capacity too small


def test_kv_packing_rule(s):
    """K/V are block-packed (B >= 8) only when the call selects at least as
    many blocks as the cache holds, or for fp32 inputs: a decode step over a
    1M paged cache carves no packed copies, a chunk of 8192 queries does, and
    the launch plan differs by exactly the two packing launches around the
    threshold."""
    big = dict(seq_kv=1 << 20, n_q_heads=64, n_kv_heads=8, head_dim=128, block_size=8,
               topk_tokens=4096, tile_q=64, page_size=64)
    packed = 2 * 8 * ((1 << 20) // 8 + 1) * 8 * 128 * 2  # K and V, one zero block per head
    dec = s.params(seq_q=1, q_offset=(1 << 20) - 1, **big)
    pre = s.params(seq_q=8192, q_offset=(1 << 20) - 8192, **big)
    assert s.workspace_bytes(dec, s.WS_SPARSE_ATTN) < (1 << 20)
    assert s.workspace_bytes(pre, s.WS_SPARSE_ATTN) >= packed
    dec32 = s.params(seq_q=1, q_offset=(1 << 20) - 1, dtype=s.FP32, **big)
    assert s.workspace_bytes(dec32, s.WS_SPARSE_ATTN) >= packed
    # 516 blocks of 8; 16 selected per query: 32 queries select 512 < 516, 40 select 640
    small = dict(n_q_heads=8, n_kv_heads=2, head_dim=128, block_size=8, topk_tokens=128,
                 tile_q=64)
    below = s.params(seq_q=32, seq_kv=4128, q_offset=4096, **small)
    above = s.params(seq_q=40, seq_kv=4136, q_offset=4096, **small)
    assert s.sgqa_prefill_plan(above)[1] - s.sgqa_prefill_plan(below)[1] == 2


def test_params_struct_matches_header(s):
    """The binding's Params fields are the header's sgqa_params fields, in order."""
    text = open(os.path.join(ROOT, "include", "sgqa.h")).read()
    body = re.search(r"typedef struct sgqa_params \{(.*?)\} sgqa_params;", text, re.S).group(1)
    fields = re.findall(r"^\s*(?:int32_t|float)\s+(\w+);", body, re.M)
    assert fields == [n for n, _ in s.Params._fields_]
    assert ctypes.sizeof(s.Params) == 4 * len(fields)


def test_batch_scales_capacity_and_plan(s):
    """batch = N covers N sequences: N times the union capacity and launches,
    the workspace of one sequence; a negative batch is rejected."""
    one = p_small(s)
    three = p_small(s, batch=3)
    assert s.union_capacity(three) == 3 * s.union_capacity(one)
    assert s.sgqa_prefill_plan(three)[1] == 3 * s.sgqa_prefill_plan(one)[1]
    assert s.sgqa_prefill_plan(three)[0] == s.sgqa_prefill_plan(one)[0]
    for w in (s.WS_INDEX_SCORES, s.WS_TOPK_UNION, s.WS_SPARSE_ATTN, s.WS_PREFILL):
        assert s.workspace_bytes(three, w) == s.workspace_bytes(one, w)
    assert s.union_capacity(p_small(s, batch=0)) == s.union_capacity(one)
    assert _call_prefill(s, p_small(s, batch=-1)) == s.ERR_INVALID_ARG


def test_debug_stall_constant_matches_header(s):
    text = open(os.path.join(ROOT, "include", "sgqa.h")).read()
    m = re.search(r"#define SGQA_DEBUG_STALL (0x[0-9a-fA-F]+)", text)
    assert m and int(m.group(1), 16) == s.DEBUG_STALL
