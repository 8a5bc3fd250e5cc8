"""kvfix_draft_rank_noalloc: the draft-rank call for callers that cannot allocate device
memory (an engine whose KV-block pool already holds nearly all of HBM, or a path that
must not pay an allocation's synchronisation).  It uses a fixed scratch buffer owned by
the library instead of a caller workspace.  This file is collected last on purpose:
the check must hold in a fresh process and after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

from cross_context_kv_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    synth.LOWRANK_70B.with_(name="noalloc_a", chunks=2, layers=3, tokens=300, kv_heads=2, q_heads=16, seed=60),
    synth.LOWRANK_70B.with_(name="noalloc_b", chunks=1, layers=5, tokens=4096, kv_heads=8, q_heads=64, seed=61),
]


def _noalloc(kvfix, k, q, layer_begin, k_rows, k_fresh=None, v_fresh=None, k_io=None, v_io=None):
    """Direct call through the C ABI; outputs are allocated here, by the caller."""
    d = kvfix.plane_desc(k)
    idx = torch.full((d.chunks, k_rows), -7, dtype=torch.int32, device=DEV)
    scores = torch.full((d.chunks, d.tokens), float("nan"), dtype=torch.float64, device=DEV)
    fd = kvfix.plane_desc(k_fresh) if k_fresh is not None else d
    p = kvfix._ptr
    st = kvfix.lib.kvfix_draft_rank_noalloc(p(k), d, p(q), int(q.shape[2]), int(q.shape[3]), int(layer_begin),
                                            int(k_rows), p(idx), p(scores), p(k_fresh), p(v_fresh), fd, p(k_io),
                                            p(v_io), kvfix._stream(k))
    return st, idx, scores


def test_noalloc_matches_draft_rank_on_consecutive_calls():
    from cross_context_kv_gb300 import kvfix
    for cfg in CASES:  # two calls in a row, different problems, one shared buffer
        inp = synth.lowrank_inputs(cfg, DEV)
        k, q = inp["x_k"], inp["q"]
        ref_k, ref_v = k.clone(), inp["x_v"].clone()
        ref_idx, ref_scores = kvfix.draft_rank(k, q, cfg.layer_begin, cfg.k_rows, inp["fresh_k"], inp["fresh_v"],
                                               ref_k, ref_v)
        got_k, got_v = k.clone(), inp["x_v"].clone()
        st, idx, scores = _noalloc(kvfix, k, q, cfg.layer_begin, cfg.k_rows, inp["fresh_k"], inp["fresh_v"],
                                   got_k, got_v)
        assert st == kvfix.OK, kvfix.lib.kvfix_last_error()
        kvfix.check_status()
        assert torch.equal(idx, ref_idx)
        np.testing.assert_allclose(scores.cpu().numpy(), ref_scores.cpu().numpy(), rtol=1e-5, atol=1e-9)
        assert torch.equal(got_k.view(torch.int16), ref_k.view(torch.int16))
        assert torch.equal(got_v.view(torch.int16), ref_v.view(torch.int16))


def test_noalloc_allocates_nothing():
    """Once the outputs exist and a first call has looked up the buffer (and loaded the
    kernels), a further call changes neither the device's free memory nor the memory
    torch's allocator holds."""
    from cross_context_kv_gb300 import kvfix
    cfg = CASES[1]
    inp = synth.lowrank_inputs(cfg, DEV)
    k_io, v_io = inp["x_k"].clone(), inp["x_v"].clone()
    d = kvfix.plane_desc(inp["x_k"])
    idx = torch.empty((d.chunks, cfg.k_rows), dtype=torch.int32, device=DEV)
    scores = torch.empty((d.chunks, d.tokens), dtype=torch.float64, device=DEV)
    p = kvfix._ptr

    def call():
        return kvfix.lib.kvfix_draft_rank_noalloc(p(inp["x_k"]), d, p(inp["q"]), int(inp["q"].shape[2]),
                                                  int(inp["q"].shape[3]), cfg.layer_begin, cfg.k_rows, p(idx),
                                                  p(scores), p(inp["fresh_k"]), p(inp["fresh_v"]), d, p(k_io),
                                                  p(v_io), kvfix._stream(k_io))
    assert call() == kvfix.OK, kvfix.lib.kvfix_last_error()
    torch.cuda.synchronize()
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    for _ in range(2):
        assert call() == kvfix.OK, kvfix.lib.kvfix_last_error()
    torch.cuda.synchronize()
    kvfix.check_status()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_reserved() == reserved0


def test_noalloc_errors_name_the_entry_point():
    """An argument error found by the draft-rank checks is reported under this entry
    point's name."""
    from cross_context_kv_gb300 import kvfix
    cfg = CASES[0]
    inp = synth.lowrank_inputs(cfg, DEV)
    d = kvfix.plane_desc(inp["x_k"])
    idx = torch.empty((d.chunks, 1), dtype=torch.int32, device=DEV)
    scores = torch.empty((d.chunks, d.tokens), dtype=torch.float64, device=DEV)
    p = kvfix._ptr
    st = kvfix.lib.kvfix_draft_rank_noalloc(p(inp["x_k"]), d, p(inp["q"]), int(inp["q"].shape[2]), 7, 1, 1,
                                            p(idx), p(scores), None, None, d, None, None, kvfix._stream(idx))
    assert st == kvfix.EINVAL  # 7 query heads is no multiple of the KV heads
    assert kvfix.lib.kvfix_last_error().startswith(b"kvfix_draft_rank_noalloc: ")


def test_noalloc_rejects_problems_beyond_the_buffer():
    """A problem whose scratch exceeds the fixed buffer is refused before anything is
    read or launched, so the descriptor may describe more rows than the buffers hold."""
    from cross_context_kv_gb300 import kvfix
    C, L, n, H, D = 2, 81, 16384, 8, 128
    row = H * D
    big = kvfix.KvDesc(C, L, n, H, D, L * n * row, n * row, row)
    assert kvfix.lib.kvfix_draft_rank_workspace_bytes(big, 1) > (64 << 20)
    k = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    q = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros(16, dtype=torch.int32, device=DEV)
    scores = torch.zeros(16, dtype=torch.float64, device=DEV)
    p = kvfix._ptr
    st = kvfix.lib.kvfix_draft_rank_noalloc(p(k), big, p(q), 2, 64, 1, 10, p(idx), p(scores), None, None, big,
                                            None, None, kvfix._stream(k))
    assert st == kvfix.EINVAL
    assert b"fixed buffer" in kvfix.lib.kvfix_last_error()
