"""GPU parity of the low-rank delta and the draft-attention row repair against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from cross_context_kv_gb300 import synth
from helpers import assert_close_kv, boundary_gap, check_index_set

pytestmark = pytest.mark.gpu
DEV = "cuda"


def kvfix():
    from cross_context_kv_gb300 import kvfix as k
    return k


SMALL_LR = [
    synth.LOWRANK_70B.with_(name="lr_small", chunks=2, layers=3, tokens=300, kv_heads=2, q_heads=16,
                            seed=40),
    synth.LOWRANK_70B.with_(name="lr_d64_r32", chunks=1, layers=2, tokens=1000, kv_heads=3, q_heads=6,
                            head_dim=64, rank=32, draft_steps=2, seed=41),
    synth.LOWRANK_70B.with_(name="lr_r64", chunks=1, layers=2, tokens=129, kv_heads=1, q_heads=8,
                            rank=64, seed=42),
]


@pytest.mark.parametrize("cfg", SMALL_LR, ids=lambda c: c.name)
def test_lowrank_apply_matches_oracle(cfg):
    inp = synth.lowrank_inputs(cfg, DEV, planes=("k",))
    out = kvfix().lowrank_apply(inp["x_k"], inp["a_k"], inp["b_k"])
    kvfix().check_status()
    ref = oracle.lowrank_apply(synth.bits(inp["x_k"]), synth.bits(inp["a_k"]), synth.bits(inp["b_k"]))
    got = synth.bits(out)
    assert_close_kv(got, ref, cfg.name)
    assert np.mean(got != ref) < 1e-2
    # in place gives the same bits
    x2 = inp["x_k"].clone()
    kvfix().lowrank_apply(x2, inp["a_k"], inp["b_k"], out=x2)
    assert torch.equal(x2.view(torch.int16), out.view(torch.int16))
    # zero factors: bit identity
    z = kvfix().lowrank_apply(inp["x_k"], torch.zeros_like(inp["a_k"]), inp["b_k"])
    assert torch.equal(z.view(torch.int16), inp["x_k"].view(torch.int16))


@pytest.mark.parametrize("cfg", SMALL_LR, ids=lambda c: c.name)
def test_draft_rank_matches_oracle(cfg):
    inp = synth.lowrank_inputs(cfg, DEV)
    kt = inp["x_k"]
    q = inp["q"]
    k_rows = cfg.k_rows
    k_io, v_io = kt.clone(), inp["x_v"].clone()
    idx, scores = kvfix().draft_rank(kt, q, cfg.layer_begin, k_rows, inp["fresh_k"], inp["fresh_v"], k_io, v_io)
    kvfix().check_status()
    kb, qb = synth.bits(kt), synth.bits(q)
    ref_scores = oracle.draft_scores(kb, qb, cfg.layer_begin)
    got_scores = scores.cpu().numpy()
    np.testing.assert_allclose(got_scores, ref_scores, rtol=1e-5, atol=1e-9)
    np.testing.assert_allclose(got_scores.sum(1), (cfg.layers - cfg.layer_begin) * cfg.draft_steps * cfg.q_heads,
                               rtol=1e-5)
    gi = idx.cpu().numpy()
    ref_idx, swapped = [], []
    for c in range(cfg.chunks):
        ri = oracle.topk(ref_scores[c], k_rows, False)
        ref_idx.append(ri)
        check_index_set(gi[c], ri, ref_scores[c], f"{cfg.name} chunk {c}")
        swapped.append(sorted(set(gi[c]) ^ set(ri)))
    # repaired planes: exactly the oracle's overwrite of its own selected rows (rows a
    # near tie swapped between the two sides are left out)
    rk = oracle.row_overwrite(kb, synth.bits(inp["fresh_k"]), np.stack(ref_idx))
    rv = oracle.row_overwrite(synth.bits(inp["x_v"]), synth.bits(inp["fresh_v"]), np.stack(ref_idx))
    gk, gv = synth.bits(k_io), synth.bits(v_io)
    for c in range(cfg.chunks):
        keep = np.setdiff1d(np.arange(cfg.tokens), swapped[c])
        assert np.array_equal(gk[c][:, keep], rk[c][:, keep])
        assert np.array_equal(gv[c][:, keep], rv[c][:, keep])


def test_draft_rank_all_rows_is_fresh_and_shift_invariance():
    cfg = SMALL_LR[0]
    inp = synth.lowrank_inputs(cfg, DEV)
    n = cfg.tokens
    k_io = inp["x_k"].clone()
    idx, scores = kvfix().draft_rank(inp["x_k"], inp["q"], 1, n, inp["fresh_k"], None, k_io, None)
    assert torch.equal(k_io.view(torch.int16), inp["fresh_k"].view(torch.int16))
    assert torch.equal(idx.cpu(), torch.arange(n, dtype=torch.int32).repeat(cfg.chunks, 1))
    # a common key shift per (layer, head), exactly representable: scores unchanged
    k_small = (torch.randint(-8, 8, inp["x_k"].shape, device=DEV) / 8.0).to(torch.bfloat16)
    shift = (torch.randint(-8, 8, (cfg.chunks, cfg.layers, 1, cfg.kv_heads, cfg.head_dim), device=DEV) / 4.0)
    k_shift = (k_small.float() + shift).to(torch.bfloat16)
    _, s0 = kvfix().draft_rank(k_small, inp["q"], 1, 0)
    _, s1 = kvfix().draft_rank(k_shift, inp["q"], 1, 0)
    np.testing.assert_allclose(s1.cpu().numpy(), s0.cpu().numpy(), rtol=2e-5)


@pytest.mark.slow
def test_full_size_lowrank_draft_parity():
    """The 70B-shaped workload in the benchmark's launch configuration: low-rank delta on
    both planes, draft ranking of the corrected keys, repair of the top 5% rows.  The
    oracle checks chunk 0 completely (scores, selection, repaired planes) and sampled
    rows of the other chunks."""
    cfg = synth.LOWRANK_70B
    inp = synth.lowrank_inputs(cfg, DEV)
    kt = kvfix().lowrank_apply(inp["x_k"], inp["a_k"], inp["b_k"])
    vt = kvfix().lowrank_apply(inp["x_v"], inp["a_v"], inp["b_v"])
    idx, scores = kvfix().draft_rank(kt, inp["q"], cfg.layer_begin, cfg.k_rows)
    kvfix().check_status()
    c = 0
    ref_kt = oracle.lowrank_apply(synth.bits(inp["x_k"][c:c + 1]), synth.bits(inp["a_k"][c:c + 1]),
                                  synth.bits(inp["b_k"][c:c + 1]))
    assert_close_kv(synth.bits(kt[c:c + 1]), ref_kt, "K~ chunk 0")
    ref_vt = oracle.lowrank_apply(synth.bits(inp["x_v"][c:c + 1]), synth.bits(inp["a_v"][c:c + 1]),
                                  synth.bits(inp["b_v"][c:c + 1]))
    assert_close_kv(synth.bits(vt[c:c + 1]), ref_vt, "V~ chunk 0")
    ref_scores = oracle.draft_scores(ref_kt, synth.bits(inp["q"][c:c + 1]), cfg.layer_begin)[0]
    np.testing.assert_allclose(scores[c].cpu().numpy(), ref_scores, rtol=1e-4)
    ri = oracle.topk(ref_scores, cfg.k_rows, False)
    swaps = check_index_set(idx[c].cpu().numpy(), ri, ref_scores, "chunk 0")
    print(f"lowrank_70b chunk 0: swaps {swaps}, boundary gap {boundary_gap(ref_scores, cfg.k_rows):.3g}")
    # other chunks: sampled rows of the low-rank output, every layer and head
    rng = np.random.default_rng(0)
    for c in range(1, cfg.chunks):
        rows = np.sort(rng.choice(cfg.tokens, 64, replace=False))
        xs = synth.bits(inp["x_k"][c:c + 1, :, rows])
        a = synth.bits(inp["a_k"][c:c + 1][:, :, :, rows])
        ref = oracle.lowrank_apply(xs, a, synth.bits(inp["b_k"][c:c + 1]))
        assert_close_kv(synth.bits(kt[c:c + 1, :, rows]), ref, f"K~ chunk {c} sampled rows")


# ------------------------------------------------------------------ fused low-rank + draft

FUSED = SMALL_LR + [
    # more (chunk, layer, head) units than resident clusters: each cluster walks several,
    # with the B/query buffers and the logits columns reused
    synth.LOWRANK_70B.with_(name="fused_many_units", chunks=2, layers=6, tokens=2100, kv_heads=4, q_heads=32,
                            seed=43),
    synth.LOWRANK_70B.with_(name="fused_layer_begin0", chunks=1, layers=3, tokens=640, kv_heads=2, q_heads=16,
                            layer_begin=0, seed=44),
]


@pytest.mark.parametrize("cfg", FUSED, ids=lambda c: c.name)
def test_lowrank_draft_equals_the_two_calls(cfg):
    """kvfix_lowrank_draft gives the bits of kvfix_lowrank_apply followed by
    kvfix_draft_rank: corrected keys, scores, selection and repaired planes."""
    inp = synth.lowrank_inputs(cfg, DEV)
    kt = kvfix().lowrank_apply(inp["x_k"], inp["a_k"], inp["b_k"])
    vt = kvfix().lowrank_apply(inp["x_v"], inp["a_v"], inp["b_v"])
    plain = kt.clone()
    ref_idx, ref_scores = kvfix().draft_rank(kt, inp["q"], cfg.layer_begin, cfg.k_rows, inp["fresh_k"],
                                             inp["fresh_v"], kt, vt)
    vt2 = kvfix().lowrank_apply(inp["x_v"], inp["a_v"], inp["b_v"])
    out, idx, scores = kvfix().lowrank_draft(inp["x_k"], inp["a_k"], inp["b_k"], inp["q"], cfg.layer_begin,
                                             cfg.k_rows, k_fresh=inp["fresh_k"], v_fresh=inp["fresh_v"], v_io=vt2)
    kvfix().check_status()
    assert torch.equal(scores, ref_scores)
    assert torch.equal(idx, ref_idx)
    assert torch.equal(out.view(torch.int16), kt.view(torch.int16))
    assert torch.equal(vt2.view(torch.int16), vt.view(torch.int16))
    # without the repair the output is the low-rank result itself; in place too
    out2, idx2, scores2 = kvfix().lowrank_draft(inp["x_k"], inp["a_k"], inp["b_k"], inp["q"], cfg.layer_begin,
                                                cfg.k_rows)
    x3 = inp["x_k"].clone()
    kvfix().lowrank_draft(x3, inp["a_k"], inp["b_k"], inp["q"], cfg.layer_begin, cfg.k_rows, out=x3)
    kvfix().check_status()
    assert torch.equal(out2.view(torch.int16), plain.view(torch.int16))
    assert torch.equal(x3.view(torch.int16), plain.view(torch.int16))
    assert torch.equal(scores2, ref_scores) and torch.equal(idx2, ref_idx)
    # against the oracle: the scores of the fused call's keys and the selection
    ref = oracle.draft_scores(synth.bits(out2), synth.bits(inp["q"]), cfg.layer_begin)
    np.testing.assert_allclose(scores2.cpu().numpy(), ref, rtol=1e-5, atol=1e-9)
    for c in range(cfg.chunks):
        check_index_set(idx2[c].cpu().numpy(), oracle.topk(ref[c], cfg.k_rows, False), ref[c], f"{cfg.name} {c}")


@pytest.mark.slow
def test_full_size_lowrank_draft_fused_equals_two_calls():
    """The 70B-shaped workload: the fused call equals the two-call sequence bit for bit
    (both planes repaired), and chunk 0's scores and selection match the oracle's."""
    cfg = synth.LOWRANK_70B
    inp = synth.lowrank_inputs(cfg, DEV)
    kt = kvfix().lowrank_apply(inp["x_k"], inp["a_k"], inp["b_k"])
    vt = kvfix().lowrank_apply(inp["x_v"], inp["a_v"], inp["b_v"])
    ref_idx, ref_scores = kvfix().draft_rank(kt, inp["q"], cfg.layer_begin, cfg.k_rows, inp["fresh_k"],
                                             inp["fresh_v"], kt, vt)
    kt2 = torch.empty_like(kt)
    vt2 = kvfix().lowrank_apply(inp["x_v"], inp["a_v"], inp["b_v"])
    _, idx, scores = kvfix().lowrank_draft(inp["x_k"], inp["a_k"], inp["b_k"], inp["q"], cfg.layer_begin, cfg.k_rows,
                                           out=kt2, k_fresh=inp["fresh_k"], v_fresh=inp["fresh_v"], v_io=vt2)
    kvfix().check_status()
    assert torch.equal(scores, ref_scores) and torch.equal(idx, ref_idx)
    assert torch.equal(kt2.view(torch.int16), kt.view(torch.int16))
    assert torch.equal(vt2.view(torch.int16), vt.view(torch.int16))
    del kt, vt, vt2, kt2
    c = 0
    ref_kt = oracle.lowrank_apply(synth.bits(inp["x_k"][c:c + 1]), synth.bits(inp["a_k"][c:c + 1]),
                                  synth.bits(inp["b_k"][c:c + 1]))
    ref_sc = oracle.draft_scores(ref_kt, synth.bits(inp["q"][c:c + 1]), cfg.layer_begin)[0]
    np.testing.assert_allclose(scores[c].cpu().numpy(), ref_sc, rtol=1e-4)
    check_index_set(idx[c].cpu().numpy(), oracle.topk(ref_sc, cfg.k_rows, False), ref_sc, "fused chunk 0")
