"""GPU parity of the repair layouts (single rows, mean-scored chunks, grown spans) and of
the counted row repair: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def kvfix():
    from cross_context_kv_gb300 import kvfix as k
    return k


def draft_like(rng, U, n):
    """Heavy-tailed positive scores, like attention masses summed over layers and heads."""
    return np.exp(2.0 * rng.standard_normal((U, n)))


CASES = [
    # (layout, chunk_tokens, budget, tau, skip)
    (0, 1, (1, 5), 0.25, True),
    (1, 64, (1, 5), 0.25, True),
    (1, 16, (1, 5), 0.25, False),
    (1, 64, (1, 20), 0.25, True),     # rho n < B at small n: skipped
    (2, 1, (1, 5), 0.25, True),
    (2, 1, (1, 5), 0.0, True),
    (2, 1, (1, 20), 2.0, True),
]


def check(scores, layout, B, budget, tau, skip):
    s = torch.as_tensor(scores, device=DEV)
    idx, cnt = kvfix().repair_layout(s, layout, B, budget, tau, skip)
    kvfix().check_status()
    ridx, rcnt = oracle.repair_layout(scores, layout, B, budget, tau, skip, max_rows=idx.shape[1])
    assert np.array_equal(cnt.cpu().numpy(), rcnt), (layout, B, budget, tau, skip)
    assert np.array_equal(idx.cpu().numpy(), ridx), (layout, B, budget, tau, skip)
    return rcnt


@pytest.mark.parametrize("n", [300, 2048, 5000])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{c[0]}_B{c[1]}_r{c[2][0]}-{c[2][1]}_t{c[3]}")
def test_layouts_match_oracle(n, case):
    rng = np.random.default_rng(n + 7 * case[0] + case[1])
    check(draft_like(rng, 3, n), *case)


def test_layouts_with_ties():
    rng = np.random.default_rng(70)
    s = np.round(rng.random((2, 1000)) * 8) / 8
    for case in CASES:
        check(s, *case)
    flat = np.ones((1, 640))
    for case in CASES:
        check(flat, *case)


def test_chunk_budgets_of_the_unit_table_on_gpu():
    rng = np.random.default_rng(71)
    s = draft_like(rng, 1, 2048)
    for unit, pct in ((1, 20.0), (16, 20.3), (64, 18.8), (256, 25.0), (1024, 50.0), (2048, 100.0)):
        cnt = check(s, 1, unit, (1, 5), 0.25, False)
        assert round(100.0 * cnt[0] / 2048, 1) == pct


def test_layout_rejects_small_max_rows():
    s = torch.rand((1, 500), dtype=torch.float64, device=DEV)
    with pytest.raises(kvfix().KvfixError):
        kvfix().repair_layout(s, 2, budget=(1, 5), max_rows=99)


def test_repair_rows_counted():
    rng = np.random.default_rng(72)
    C, L, n, H, D = 3, 2, 400, 2, 64
    kv = torch.randn((C, L, n, H, D), device=DEV).to(torch.bfloat16)
    vv = torch.randn_like(kv)
    kf = torch.randn_like(kv)
    vf = torch.randn_like(kv)
    scores = torch.as_tensor(draft_like(rng, C, n), device=DEV)
    idx, cnt = kvfix().repair_layout(scores, 1, 64, (1, 4), skip_rule=False)
    assert len(set(cnt.tolist())) >= 1
    k2, v2 = kv.clone(), vv.clone()
    kvfix().repair_rows(k2, v2, kf, vf, idx, cnt)
    kvfix().check_status()
    for c in range(C):
        rows = idx[c, :cnt[c]].long()
        keep = torch.ones(n, dtype=torch.bool, device=DEV)
        keep[rows] = False
        assert torch.equal(k2[c][:, rows], kf[c][:, rows]) and torch.equal(v2[c][:, rows], vf[c][:, rows])
        assert torch.equal(k2[c][:, keep], kv[c][:, keep]) and torch.equal(v2[c][:, keep], vv[c][:, keep])


@pytest.mark.slow
def test_full_size_layouts():
    """Four 16384-row units (the draft workload's chunk length), every layout."""
    rng = np.random.default_rng(73)
    s = draft_like(rng, 4, 16384)
    for case in CASES + [(1, 64, (1, 20), 0.25, True), (2, 1, (1, 20), 0.25, True)]:
        check(s, *case)


def test_layout_edges():
    rng = np.random.default_rng(74)
    one = draft_like(rng, 2, 1)
    for case in ((0, 1, (1, 1), 0.25, True), (2, 1, (1, 1), 0.25, True), (1, 64, (1, 1), 0.25, False)):
        check(one, *case)
    s = draft_like(rng, 3, 700)
    for case in ((0, 1, (0, 1), 0.25, True), (2, 1, (0, 1), 0.25, True), (1, 1024, (1, 5), 0.25, False),
                 (1, 1024, (1, 5), 0.25, True), (2, 1, (1, 1), 0.5, True), (1, 1, (1, 1), 0.25, True)):
        check(s, *case)
