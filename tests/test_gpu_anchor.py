"""GPU parity of the anchor-pool correction (reliability gate, token weights, weighted
low-rank correction) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from cross_context_kv_gb300 import synth
from helpers import assert_close_kv

pytestmark = pytest.mark.gpu
DEV = "cuda"


def kvfix():
    from cross_context_kv_gb300 import kvfix as k
    return k


SMALL = [
    synth.ANCHOR_8B.with_(name="anchor_small", segments=2, anchors=3, layers=2, tokens=200, kv_heads=2,
                          head_dim=64, rank=16, seed=60),
    synth.ANCHOR_8B.with_(name="anchor_ten", segments=1, anchors=10, layers=2, tokens=300, kv_heads=8,
                          head_dim=128, rank=32, seed=61),
    synth.ANCHOR_8B.with_(name="anchor_sixteen", segments=2, anchors=16, layers=1, tokens=130, kv_heads=4,
                          head_dim=64, rank=16, seed=62),
    # three heads: the correction's last head group is short (two heads per MMA, then one)
    synth.ANCHOR_8B.with_(name="anchor_ragged_heads", segments=1, anchors=5, layers=2, tokens=200, kv_heads=3,
                          head_dim=128, rank=32, seed=64),
    # rank 64, six heads of 64: groups of four heads, then two
    synth.ANCHOR_8B.with_(name="anchor_rank64", segments=2, anchors=4, layers=1, tokens=150, kv_heads=6,
                          head_dim=64, rank=64, seed=65),
    # rank 64, head 128, seven anchors: one head per MMA group (shared memory)
    synth.ANCHOR_8B.with_(name="anchor_rank64_wide", segments=1, anchors=7, layers=1, tokens=140, kv_heads=2,
                          head_dim=128, rank=64, seed=66),
]


def compose(cfg, inp):
    """Source planes: the base state of the segment's matching anchor plus the noise draw
    (input construction, float32 on the device)."""
    out = {}
    for p in ("k", "v"):
        src = torch.empty_like(inp[f"noise_{p}"])
        for c in range(cfg.segments):
            v = inp["match"][c]
            rec = torch.matmul(inp[f"a_c_{p}"][c, v].float(), inp[f"b_ct_{p}"][c, v].float().transpose(-1, -2))
            src[c] = (rec.view(src[c].shape) + inp[f"noise_{p}"][c].float()).to(torch.bfloat16)
        out[p] = src
    return out


def factors(inp):
    return {k: inp[k] for k in ("a_c_k", "b_ct_k", "a_c_v", "b_ct_v", "a_d_k", "b_dt_k", "a_d_v", "b_dt_v")}


def flat(x):
    """[C][L][n][H][D] -> host bits [C][L][n][H*D]."""
    b = synth.bits(x)
    return b.reshape(b.shape[0], b.shape[1], b.shape[2], -1)


def check_gate(got, ref, tau, what):
    d, g, hbar, acc = (t.cpu().numpy() for t in got)
    rd, rg, rh, racc = ref
    np.testing.assert_allclose(d, rd, rtol=1e-5, err_msg=what)
    np.testing.assert_allclose(g, rg, atol=1e-5, err_msg=what)
    np.testing.assert_allclose(hbar, rh, atol=1e-5, err_msg=what)
    near = np.abs(rh - tau) < 1e-5
    assert np.array_equal(acc.astype(bool)[~near], racc[~near]), what


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_anchor_gate_matches_oracle(cfg):
    inp = synth.anchor_inputs(cfg, DEV)
    src = compose(cfg, inp)
    for k in (cfg.tokens, 77):
        got = kvfix().anchor_gate(src["v"], inp["a_c_v"], inp["b_ct_v"], k, tau=cfg.tau)
        kvfix().check_status()
        ref = oracle.anchor_gate(flat(src["v"]), synth.bits(inp["a_c_v"]), synth.bits(inp["b_ct_v"]), k, tau=cfg.tau)
        check_gate(got, ref, cfg.tau, f"{cfg.name} k={k}")


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_anchor_correct_matches_oracle(cfg):
    inp = synth.anchor_inputs(cfg, DEV)
    src = compose(cfg, inp)
    ok, ov, wk, wv = kvfix().anchor_correct(src["k"], src["v"], factors(inp), inp["delta"], cfg.rope_base)
    kvfix().check_status()
    H = cfg.kv_heads
    for p, got_w, got_o, rot in (("k", wk, ok, True), ("v", wv, ov, False)):
        x = flat(src[p])
        rw = oracle.anchor_weights(x, synth.bits(inp[f"a_c_{p}"]), synth.bits(inp[f"b_ct_{p}"]))
        np.testing.assert_allclose(got_w.cpu().numpy(), rw, rtol=1e-4, atol=2e-6, err_msg=f"{cfg.name} w_{p}")
        assert (rw.max(-1) / rw.min(-1)).mean() > 1.5   # the weights are not flat
        ro = oracle.anchor_correct(x, synth.bits(inp[f"a_d_{p}"]), synth.bits(inp[f"b_dt_{p}"]), rw, H,
                                   inp["delta"].cpu().numpy(), cfg.rope_base, rot)
        got = flat(got_o)
        assert_close_kv(got, ro, f"{cfg.name} out_{p}")
        # the delta term is small next to the source: compare it on its own scale too
        base = oracle.anchor_correct(x, np.zeros_like(synth.bits(inp[f"a_d_{p}"])), synth.bits(inp[f"b_dt_{p}"]),
                                     rw, H, inp["delta"].cpu().numpy(), cfg.rope_base, rot)
        dref = oracle.bf16_decode(ro) - oracle.bf16_decode(base)
        dgot = oracle.bf16_decode(got) - oracle.bf16_decode(base)
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(oracle.bf16_decode(ro)), 1e-30))) - 7)
        assert (np.abs(dgot - dref) <= 1.01 * ulp + 1e-2 * np.abs(dref).max()).all(), f"{cfg.name} delta_{p}"


def test_anchor_rejected_segments_are_untouched():
    cfg = SMALL[0]
    inp = synth.anchor_inputs(cfg, DEV)
    src = compose(cfg, inp)
    _, _, _, acc = kvfix().anchor_gate(src["v"], inp["a_c_v"], inp["b_ct_v"], cfg.tokens, tau=-1.0)
    assert not acc.any()                                   # nothing passes a negative threshold
    accept = torch.tensor([1, 0], dtype=torch.int32, device=DEV)
    ok = torch.full_like(src["k"], 7.0)
    ov = torch.full_like(src["v"], 7.0)
    wk = torch.full((cfg.segments, cfg.layers, cfg.tokens, cfg.anchors), -1.0, device=DEV)
    wv = wk.clone()
    kvfix().anchor_correct(src["k"], src["v"], factors(inp), inp["delta"], cfg.rope_base, accept=accept,
                           out_k=ok, out_v=ov, w_k=wk, w_v=wv)
    kvfix().check_status()
    assert (ok[1] == 7.0).all() and (ov[1] == 7.0).all() and (wk[1] == -1.0).all() and (wv[1] == -1.0).all()
    full_k, full_v, _, _ = kvfix().anchor_correct(src["k"], src["v"], factors(inp), inp["delta"], cfg.rope_base)
    assert torch.equal(ok[0].view(torch.int16), full_k[0].view(torch.int16))
    assert torch.equal(ov[0].view(torch.int16), full_v[0].view(torch.int16))


def test_anchor_correct_in_place():
    cfg = SMALL[1]
    inp = synth.anchor_inputs(cfg, DEV)
    src = compose(cfg, inp)
    ok, ov, _, _ = kvfix().anchor_correct(src["k"], src["v"], factors(inp), inp["delta"], cfg.rope_base)
    k2, v2 = src["k"].clone(), src["v"].clone()
    kvfix().anchor_correct(k2, v2, factors(inp), inp["delta"], cfg.rope_base, out_k=k2, out_v=v2)
    kvfix().check_status()
    assert torch.equal(k2.view(torch.int16), ok.view(torch.int16))
    assert torch.equal(v2.view(torch.int16), ov.view(torch.int16))


@pytest.mark.slow
def test_full_size_anchor_sampled():
    """Llama-8B-shaped segments, the benchmark's launch configuration: the gate over a
    256-row prefix against the oracle, the full gate deterministic and accepting, and the
    weights and outputs of sampled tokens against the oracle on those rows."""
    cfg = synth.ANCHOR_8B
    inp = synth.anchor_inputs(cfg, DEV)
    src = compose(cfg, inp)
    k = 256
    got = kvfix().anchor_gate(src["v"], inp["a_c_v"], inp["b_ct_v"], k, tau=cfg.tau)
    ref = oracle.anchor_gate(flat(src["v"][:, :, :k]), synth.bits(inp["a_c_v"][:, :, :, :k]),
                             synth.bits(inp["b_ct_v"]), k, tau=cfg.tau)
    check_gate(got, ref, cfg.tau, "prefix 256")
    g1 = kvfix().anchor_gate(src["v"], inp["a_c_v"], inp["b_ct_v"], cfg.tokens, tau=cfg.tau)
    g2 = kvfix().anchor_gate(src["v"], inp["a_c_v"], inp["b_ct_v"], cfg.tokens, tau=cfg.tau)
    assert all(torch.equal(a, b) for a, b in zip(g1[:2], g2[:2])) and g1[3].all()
    ok, ov, wk, wv = kvfix().anchor_correct(src["k"], src["v"], factors(inp), inp["delta"], cfg.rope_base,
                                            accept=g1[3])
    kvfix().check_status()
    rng = np.random.default_rng(8)
    ts = torch.as_tensor(np.sort(rng.choice(cfg.tokens, 24, replace=False)), device=DEV)
    for p, got_w, got_o, rot in (("k", wk, ok, True), ("v", wv, ov, False)):
        x = flat(src[p][:, :, ts])
        a_c = synth.bits(inp[f"a_c_{p}"][:, :, :, ts])
        rw = oracle.anchor_weights(x, a_c, synth.bits(inp[f"b_ct_{p}"]))
        np.testing.assert_allclose(got_w[:, :, ts].cpu().numpy(), rw, rtol=1e-4, atol=2e-6)
        ro = oracle.anchor_correct(x, synth.bits(inp[f"a_d_{p}"][:, :, :, ts]), synth.bits(inp[f"b_dt_{p}"]), rw,
                                   cfg.kv_heads, inp["delta"].cpu().numpy(), cfg.rope_base, rot)
        assert_close_kv(flat(got_o[:, :, ts]), ro, f"sampled out_{p}")


def test_single_anchor_gate_rejects_and_weights_are_one():
    cfg = SMALL[0].with_(anchors=1, seed=63)
    inp = synth.anchor_inputs(cfg, DEV)
    src = compose(cfg, inp)
    d, g, hbar, acc = kvfix().anchor_gate(src["v"], inp["a_c_v"], inp["b_ct_v"], cfg.tokens, tau=1.0)
    kvfix().check_status()
    assert not acc.any() and torch.isnan(hbar).all() and (g == 1.0).all()
    ok, ov, wk, wv = kvfix().anchor_correct(src["k"], src["v"], factors(inp), inp["delta"], cfg.rope_base)
    kvfix().check_status()
    assert (wk == 1.0).all() and (wv == 1.0).all()
    ro = oracle.anchor_correct(flat(src["v"]), synth.bits(inp["a_d_v"]), synth.bits(inp["b_dt_v"]),
                               np.ones((cfg.segments, cfg.layers, cfg.tokens, 1)), cfg.kv_heads,
                               inp["delta"].cpu().numpy(), cfg.rope_base, False)
    assert_close_kv(flat(ov), ro, "single anchor out_v")


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_gate_correct_in_one_pass(cfg):
    """The fused call gives the gate of kvfix_anchor_gate (to rounding, against the oracle)
    and the outputs of kvfix_anchor_correct for accepted segments, untouched ones for the
    rejected."""
    inp = synth.anchor_inputs(cfg, DEV)
    src = compose(cfg, inp)
    for k, tau in ((cfg.tokens, cfg.tau), (77, cfg.tau), (cfg.tokens, -1.0)):
        ok0 = torch.full_like(src["k"], 3.0)
        ov0 = torch.full_like(src["v"], 3.0)
        ok, ov, wk, wv, d, g, hbar, acc = kvfix().anchor_gate_correct(
            src["k"], src["v"], factors(inp), k, inp["delta"], cfg.rope_base, tau=tau, out_k=ok0, out_v=ov0)
        kvfix().check_status()
        ref = oracle.anchor_gate(flat(src["v"]), synth.bits(inp["a_c_v"]), synth.bits(inp["b_ct_v"]), k, tau=tau)
        check_gate((d, g, hbar, acc), ref, tau, f"{cfg.name} k={k}")
        rk, rv, rwk, rwv = kvfix().anchor_correct(src["k"], src["v"], factors(inp), inp["delta"], cfg.rope_base)
        assert torch.equal(wk, rwk) and torch.equal(wv, rwv)
        for c in range(cfg.segments):
            if acc[c]:
                assert torch.equal(ok[c].view(torch.int16), rk[c].view(torch.int16))
                assert torch.equal(ov[c].view(torch.int16), rv[c].view(torch.int16))
            else:
                assert (ok[c] == 3.0).all() and (ov[c] == 3.0).all()
    g1 = kvfix().anchor_gate_correct(src["k"], src["v"], factors(inp), cfg.tokens, inp["delta"], cfg.rope_base)
    g2 = kvfix().anchor_gate_correct(src["k"], src["v"], factors(inp), cfg.tokens, inp["delta"], cfg.rope_base)
    assert torch.equal(g1[4], g2[4])                 # deterministic distances


def test_persistent_kernels_walk_many_units():
    """More (row tile, layer, plane, segment) units than SMs, so every CTA of the
    persistent distance and apply kernels walks several units and skips rejected
    segments: the outputs of the accepted segment equal a call on that segment alone,
    bit for bit, and the rejected segment's outputs and weights keep their fill."""
    cfg = synth.ANCHOR_8B.with_(name="anchor_many", segments=2, anchors=4, layers=4, tokens=4096, kv_heads=2,
                                head_dim=128, rank=16, seed=64)
    inp = synth.anchor_inputs(cfg, DEV)
    src = compose(cfg, inp)
    fac = factors(inp)
    # a temperature on the scale of the gate's distances, so that the entropies of the two
    # segments lie strictly between 0 and 1 (at T = 1 each segment matches one anchor so
    # closely that both entropies are 0)
    d0, _, _, _ = kvfix().anchor_gate(src["v"], inp["a_c_v"], inp["b_ct_v"], cfg.tokens, tau=cfg.tau)
    T = float(d0.mean().item())
    ref = [kvfix().anchor_correct(src["k"][c:c + 1], src["v"][c:c + 1], {k: v[c:c + 1] for k, v in fac.items()},
                                  inp["delta"][c:c + 1], cfg.rope_base, temperature=T) for c in range(cfg.segments)]
    ok = torch.full_like(src["k"], 7.0)
    ov = torch.full_like(src["v"], 7.0)
    wk = torch.full((cfg.segments, cfg.layers, cfg.tokens, cfg.anchors), -1.0, device=DEV)
    wv = wk.clone()
    accept = torch.tensor([1, 0], dtype=torch.int32, device=DEV)
    kvfix().anchor_correct(src["k"], src["v"], fac, inp["delta"], cfg.rope_base, temperature=T, accept=accept,
                           out_k=ok, out_v=ov, w_k=wk, w_v=wv)
    kvfix().check_status()
    assert torch.equal(ok[0].view(torch.int16), ref[0][0][0].view(torch.int16))
    assert torch.equal(ov[0].view(torch.int16), ref[0][1][0].view(torch.int16))
    assert torch.equal(wk[0], ref[0][2][0]) and torch.equal(wv[0], ref[0][3][0])
    assert (ok[1] == 7.0).all() and (ov[1] == 7.0).all() and (wk[1] == -1.0).all() and (wv[1] == -1.0).all()
    # the one-pass call with a threshold between the two segments' entropies: one passes
    _, _, hbar, _ = kvfix().anchor_gate(src["v"], inp["a_c_v"], inp["b_ct_v"], cfg.tokens, temperature=T,
                                        tau=cfg.tau)
    h = hbar.cpu().numpy()
    assert 0.0 < h.min() < h.max() < 1.0
    tau = float((h[0] + h[1]) / 2)
    ok2 = torch.full_like(src["k"], 3.0)
    ov2 = torch.full_like(src["v"], 3.0)
    res = kvfix().anchor_gate_correct(src["k"], src["v"], fac, cfg.tokens, inp["delta"], cfg.rope_base, temperature=T,
                                      tau=tau, out_k=ok2, out_v=ov2)
    kvfix().check_status()
    acc = res[7].cpu().numpy().astype(bool)
    assert acc.sum() == 1
    for c in range(cfg.segments):
        if acc[c]:
            assert torch.equal(ok2[c].view(torch.int16), ref[c][0][0].view(torch.int16))
            assert torch.equal(ov2[c].view(torch.int16), ref[c][1][0].view(torch.int16))
        else:
            assert (ok2[c] == 3.0).all() and (ov2[c] == 3.0).all()
