"""Shared test helpers: tolerance and near-tie checks, synthetic inputs composed by the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from cross_context_kv_gb300 import synth

# Tolerances for corrected K/V (bf16 outputs, float accumulation): max-abs error at most
# 1e-2 of the reference's largest magnitude, and pooled mean relative error at most 2e-3.
MAX_ABS_FRAC = 1e-2
MEAN_REL = 2e-3
NEAR_TIE_REL = 1e-5


def assert_close_kv(got_bits, ref_bits, what=""):
    got = oracle.bf16_decode(np.ascontiguousarray(got_bits))
    ref = oracle.bf16_decode(np.ascontiguousarray(ref_bits))
    err = np.abs(got - ref)
    scale = np.abs(ref).max() if ref.size else 0.0
    assert err.max(initial=0.0) <= MAX_ABS_FRAC * scale + 1e-30, \
        f"{what}: max|err| {err.max():.4g} > {MAX_ABS_FRAC} * {scale:.4g}"
    denom = np.abs(ref).sum()
    if denom > 0:
        rel = err.sum() / denom
        assert rel <= MEAN_REL, f"{what}: mean relative error {rel:.3g} > {MEAN_REL}"
    return err


def check_index_set(got, ref, scores, what=""):
    """Equal sets pass.  Otherwise every swapped pair must be a near tie (< 1e-5 relative)
    in the oracle's scores.  Returns the number of swapped pairs."""
    got = np.asarray(got)
    ref = np.asarray(ref)
    assert got.shape == ref.shape, f"{what}: shapes {got.shape} vs {ref.shape}"
    assert np.all(np.diff(got) > 0) if got.size > 1 else True, f"{what}: GPU indices not ascending"
    sg, sr = set(got.tolist()), set(ref.tolist())
    extra, missing = sorted(sg - sr), sorted(sr - sg)
    for i, j in zip(extra, missing):
        si, sj = float(scores[i]), float(scores[j])
        rel = abs(si - sj) / max(abs(si), abs(sj), 1e-300)
        assert rel < NEAR_TIE_REL, f"{what}: swap {i}<->{j} not a near tie ({rel:.3g})"
    return len(extra)


def boundary_gap(scores, b):
    """Relative gap between the b-th and (b+1)-th largest scores (inf if none)."""
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    if b <= 0 or b >= s.size:
        return float("inf")
    return float((s[b - 1] - s[b]) / max(abs(s[b - 1]), 1e-300))


def repair_inputs(cfg: synth.RepairConfig, device):
    """Draws on `device`, fresh planes composed by the oracle on the host.
    Returns dict of torch tensors on `device` plus host bit arrays."""
    reuse = synth.repair_reuse(cfg, device)
    rk, rv = synth.bits(reuse["k_reuse"]), synth.bits(reuse["v_reuse"])
    delta = reuse["delta"].cpu().numpy()
    R, A = cfg.chunks, cfg.agents
    fk = np.empty((A * R,) + rk.shape[1:], np.uint16)
    fv = np.empty_like(fk)
    for u in range(A * R):
        res = synth.repair_residual(cfg, u, device)
        r = u % R
        fk[u:u + 1] = oracle.compose_fresh(rk[r:r + 1], res["mu_k"][None].cpu().numpy(),
                                           res["xi_k"][None].cpu().numpy(), delta[u:u + 1], 1,
                                           cfg.rope_base, True)
        fv[u:u + 1] = oracle.compose_fresh(rv[r:r + 1], res["mu_v"][None].cpu().numpy(),
                                           res["xi_v"][None].cpu().numpy(), delta[u:u + 1], 1,
                                           cfg.rope_base, False)
    return {"k_reuse": reuse["k_reuse"], "v_reuse": reuse["v_reuse"], "delta": reuse["delta"],
            "k_fresh": synth.from_bits(fk, device), "v_fresh": synth.from_bits(fv, device),
            "rk": rk, "rv": rv, "fk": fk, "fv": fv, "delta_np": delta}
