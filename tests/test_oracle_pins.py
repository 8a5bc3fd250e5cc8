"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test ties one oracle function to something other than its own formula: values
printed on the pages (tests/golden/), closed forms, invariants of the mathematics,
special cases that reduce to a library routine, or brute force on tiny inputs.  The
cases are chosen so that a plausible slip (a dropped term, a flipped sign, a wrong
index, a transposed operand) breaks at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = [float(v) for v in vals]
    return rows


def _bf16_bits(x):
    return oracle.bf16_encode(np.asarray(x, dtype=np.float64))


# ------------------------------------------------------------------ bf16

def test_bf16_encode_matches_torch_rounding():
    """The oracle's double->float->bf16 rounding equals torch's float->bf16 cast
    (round to nearest even) on random values, exact ties and specials."""
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
        # exact ties between two bf16 neighbours: lower half = 0x8000
        (np.frombuffer((rng.integers(0, 2**15, 2000, dtype=np.uint32) << 16 | 0x8000)
                       .astype(np.uint32).tobytes(), dtype=np.float32)).astype(np.float64),
        [0.0, -0.0, np.inf, -np.inf, 3.3895313892515355e38, 1e-45, -1e-45],
    ])
    x = x[np.isfinite(x.astype(np.float32)) | np.isinf(x)]
    ours = oracle.bf16_encode(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(ours, ref.view(np.uint16))


def test_bf16_decode_is_exact():
    h = np.arange(0, 2**16, dtype=np.uint16)
    h = h[(h & 0x7F80) != 0x7F80]  # finite patterns
    d = oracle.bf16_decode(h)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(d, ref)
    assert np.array_equal(oracle.bf16_encode(d), h)


# ------------------------------------------------------------------ RoPE

def test_rope_theta_closed_form():
    for base, D in ((1e4, 64), (5e5, 128), (1e6, 128)):
        th = oracle.rope_theta(base, D)
        i = np.arange(D // 2)
        np.testing.assert_allclose(th, np.power(base, -2.0 * i / D), rtol=1e-15)
        assert th[0] == 1.0


def test_rotation_matches_complex_multiplication():
    """Rotate-half RoPE is multiplication of (x_i + i x_{i+D/2}) by exp(i delta theta_i)."""
    rng = np.random.default_rng(1)
    D, base = 128, 5e5
    x = rng.standard_normal((7, D))
    for delta in (0, 1, 137, 4321, 8000, -55):
        y = oracle.rotate_f64(x, delta, base)
        th = np.power(base, -2.0 * np.arange(D // 2) / D)
        z = (x[:, : D // 2] + 1j * x[:, D // 2:]) * np.exp(1j * delta * th)
        np.testing.assert_allclose(y[:, : D // 2], z.real, atol=1e-12)
        np.testing.assert_allclose(y[:, D // 2:], z.imag, atol=1e-12)


def test_rotation_composes_and_inverts():
    rng = np.random.default_rng(2)
    D, base = 64, 1e4
    x = rng.standard_normal((5, D))
    for p, q in ((3, 5), (137, 1000), (7999, 1), (-40, 40)):
        a = oracle.rotate_f64(oracle.rotate_f64(x, p, base), q, base)
        b = oracle.rotate_f64(x, p + q, base)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    back = oracle.rotate_f64(oracle.rotate_f64(x, 321, base), -321, base)
    np.testing.assert_allclose(back, x, atol=1e-12)
    y = oracle.rotate_f64(x, 77, base)
    pair_in = x[:, :32] ** 2 + x[:, 32:] ** 2
    pair_out = y[:, :32] ** 2 + y[:, 32:] ** 2
    np.testing.assert_allclose(pair_out, pair_in, rtol=1e-12)


def test_rerope_zero_shift_is_bit_identity_and_matches_rotation():
    rng = np.random.default_rng(3)
    k = _bf16_bits(rng.standard_normal((2, 3, 8, 2, 64)))
    assert np.array_equal(oracle.rerope(k, [0, 0], 1e4), k)
    out = oracle.rerope(k, [137, 9], 1e4)
    for c, delta in enumerate((137, 9)):
        y = oracle.rotate_f64(oracle.bf16_decode(k[c]), delta, 1e4)
        assert np.array_equal(out[c], _bf16_bits(y))


# ------------------------------------------------------------------ scores

def test_scores_constant_value_offset_closed_form():
    """Values (no rotation): fresh = reuse + c exactly -> d = |c| sqrt(H D)."""
    rng = np.random.default_rng(4)
    R, n, H, D = 1, 9, 2, 8
    reuse = _bf16_bits(rng.integers(-8, 8, (R, n, H, D)).astype(np.float64))
    c = 0.375
    fresh = _bf16_bits(oracle.bf16_decode(reuse) + c)
    d = oracle.scores(reuse, fresh, [5], 1, 1e4, rotate_keys=False)
    np.testing.assert_allclose(d, np.full((1, n), c * math.sqrt(H * D)), rtol=1e-15)


def test_scores_rotation_invariant_form():
    """||fresh - R x|| = ||R^-1 fresh - x|| for a rotation R (orthogonality)."""
    rng = np.random.default_rng(5)
    A, R, n, H, D = 2, 1, 6, 3, 16
    reuse = _bf16_bits(rng.standard_normal((R, n, H, D)))
    fresh = _bf16_bits(rng.standard_normal((A * R, n, H, D)))
    delta = np.array([11, 300], np.int32)
    d = oracle.scores(reuse, fresh, delta, A, 1e4, rotate_keys=True)
    for a in range(A):
        back = oracle.rotate_f64(oracle.bf16_decode(fresh[a]), -int(delta[a]), 1e4)
        ref = np.sqrt(((back - oracle.bf16_decode(reuse[0])) ** 2).sum(axis=(1, 2)))
        np.testing.assert_allclose(d[a], ref, rtol=1e-12)


def test_scores_one_hot_difference():
    """fresh equal to the rotated cache except one element raised by 1 (away from the
    rotated value) scores ~1 on that token and ~rounding noise elsewhere."""
    rng = np.random.default_rng(6)
    n, H, D = 5, 2, 8
    reuse = _bf16_bits(rng.standard_normal((1, n, H, D)))
    rot = oracle.rotate_f64(oracle.bf16_decode(reuse), 50, 1e4)
    f = rot.copy()
    f[0, 3, 1, 5] += 1.0
    fresh = _bf16_bits(f)
    d = oracle.scores(reuse, fresh, [50], 1, 1e4, rotate_keys=True)[0]
    bound = math.sqrt(H * D) * 2.0 ** -8 * np.abs(rot).max() + 2.0 ** -8 * 4
    assert abs(d[3] - 1.0) < bound
    assert np.all(np.delete(d, 3) < bound)


# ------------------------------------------------------------------ top-b

def _brute_top(keys, b):
    """The unique b-subset whose every member precedes every non-member in the order
    (key desc, index asc), by enumeration."""
    n = len(keys)
    found = []
    for S in itertools.combinations(range(n), b):
        inside = set(S)
        ok = all((keys[i] > keys[j]) or (keys[i] == keys[j] and i < j)
                 for i in inside for j in range(n) if j not in inside)
        if ok:
            found.append(list(S))
    assert len(found) == 1
    return found[0]


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(7)
    for trial in range(60):
        n = int(rng.integers(1, 11))
        b = int(rng.integers(0, n + 1))
        keys = rng.integers(0, 4, n).astype(np.float64)  # many ties
        if trial % 2:
            keys = rng.standard_normal(n)
        got = oracle.topk(keys, b, keys_as_float=False)
        assert list(got) == _brute_top(list(keys), b)


def test_topk_all_equal_and_extremes():
    keys = np.full(40, 0.5)
    assert list(oracle.topk(keys, 7, False)) == list(range(7))
    assert list(oracle.topk(keys, 0, False)) == []
    assert list(oracle.topk(np.arange(40.0), 40, False)) == list(range(40))


def test_topk_matches_lexsort():
    rng = np.random.default_rng(8)
    keys = rng.standard_normal(3000).round(2)
    b = 455
    order = np.lexsort((np.arange(keys.size), -keys))
    assert np.array_equal(oracle.topk(keys, b, False), np.sort(order[:b]))


def test_topk_float_decision():
    """keys_as_float ranks by the binary32 value: keys equal in float tie to the lower index."""
    keys = np.array([1.0 + 2.0 ** -40, 1.0, 0.5])
    assert list(oracle.topk(keys, 1, False)) == [0]
    assert list(oracle.topk(keys[::-1].copy(), 1, True)) == [1]


# ---------------------------------------------------------- mean correction

def test_worked_example_scalar():
    g = _golden("agentkvshift_worked_example.txt")
    reused = [g[t][0] for t in "ABC"]
    weight = [g[t][2] for t in "ABC"]
    mu, out = oracle.correct_with_weights(g["probe_residuals"], reused, weight)
    assert abs(mu - g["estimated_offset"][0]) < 1e-12
    np.testing.assert_allclose(out, [g[t][3] for t in "ABC"], atol=1e-12)
    # residual of token A drops from 2.1 to 0.1 (target 12.1)
    assert abs((g["A"][1] - out[0]) - 0.1) < 1e-12


def test_worked_example_through_tensor_path():
    """The same example through the full oracle path on the value plane: probes carry
    residuals bf16(2.2) = 2.203125 and bf16(1.8) = 1.796875, whose mean is exactly 2."""
    g = _golden("agentkvshift_worked_example.txt")
    n, H, D = 5, 1, 2
    reuse = np.zeros((1, 1, n, H, D))
    reuse[0, 0, 2:, 0, :] = np.array([g["A"][0], g["B"][0], g["C"][0]])[:, None]
    fresh = reuse.copy()
    fresh[0, 0, 0] += g["probe_residuals"][0]
    fresh[0, 0, 1] += g["probe_residuals"][1]
    fresh[0, 0, 2:, 0, :] = np.array([g["A"][1], g["B"][1], g["C"][1]])[:, None]
    w = np.array([[1.0, 1.0, g["A"][2], g["B"][2], g["C"][2]]])
    out, mu = oracle.mean_correct(_bf16_bits(reuse), _bf16_bits(fresh), [0], 1, 1e4, False,
                                  np.array([[0, 1]]), w)
    assert np.all(mu == 2.0)
    got = oracle.bf16_decode(out)[0, 0, :, 0, 0]
    assert list(got[2:]) == [12.0, 21.0, 30.25]  # 30.2 rounds to the bf16 value 30.25
    assert np.array_equal(out[0, 0, :2], _bf16_bits(fresh)[0, 0, :2])


def _exact_problem(rng, A, R, L, n, H, D):
    reuse = rng.integers(-16, 16, (R, L, n, H, D)).astype(np.float64) / 4.0
    mu = rng.integers(-8, 8, (A * R, L, H, D)).astype(np.float64) / 8.0
    return reuse, mu


def test_constant_offset_recovered_exactly():
    """A pure per-(layer, head) offset with unit weights is recovered bit for bit."""
    rng = np.random.default_rng(9)
    A, R, L, n, H, D = 2, 1, 3, 20, 2, 8
    reuse, mu = _exact_problem(rng, A, R, L, n, H, D)
    mu[np.abs(mu).sum(axis=(2, 3)) == 0] = 0.5
    fresh = reuse[np.zeros(A * R, int)] + mu[:, :, None, :, :]
    rb, fb = _bf16_bits(reuse), _bf16_bits(fresh)
    assert np.array_equal(oracle.bf16_decode(fb), fresh)
    for rotate, delta in ((False, [9, 4]), (True, [0, 0])):
        d = oracle.scores(rb[:, 1], fb[:, 1], delta, A, 1e4, rotate)
        w = np.minimum(d, 1.0)
        assert np.all(w == 1.0)
        idx = np.stack([oracle.topk(d[a], 4, True) for a in range(A)])
        out, mu_hat = oracle.mean_correct(rb, fb, delta, A, 1e4, rotate, idx, w)
        assert np.array_equal(mu_hat, mu)
        assert np.array_equal(out, fb)


def test_all_probes_reproduce_fresh():
    """b = n: every row is a probe and the output is the fresh cache bit for bit."""
    rng = np.random.default_rng(10)
    R, L, n, H, D = 1, 2, 12, 2, 16
    reuse = _bf16_bits(rng.standard_normal((R, L, n, H, D)))
    fresh = _bf16_bits(rng.standard_normal((R, L, n, H, D)))
    idx = np.arange(n)[None]
    out, _ = oracle.mean_correct(reuse, fresh, [77], 1, 1e4, True, idx, np.ones((1, n)))
    assert np.array_equal(out, fresh)


def test_no_probes_is_plain_rerope():
    rng = np.random.default_rng(11)
    R, L, n, H, D = 1, 2, 12, 2, 16
    reuse = _bf16_bits(rng.standard_normal((R, L, n, H, D)))
    fresh = _bf16_bits(rng.standard_normal((R, L, n, H, D)))
    out, mu = oracle.mean_correct(reuse, fresh, [77], 1, 1e4, True, np.zeros((1, 0), np.int32),
                                  np.ones((1, n)))
    assert np.all(mu == 0)
    assert np.array_equal(out, oracle.rerope(reuse, [77], 1e4))


def test_error_identity_unit_weights():
    """With unit weights, corrected - fresh = e - xi_j on non-probes, e = mu_hat - mu
    (AgentKVShift, the error identity of the idealised analysis)."""
    rng = np.random.default_rng(12)
    L, n, H, D = 2, 30, 1, 4
    reuse, mu = _exact_problem(rng, 1, 1, L, n, H, D)
    xi = rng.integers(-4, 4, (1, L, n, H, D)).astype(np.float64) / 16.0
    fresh = reuse + mu[:, :, None] + xi
    rb, fb = _bf16_bits(reuse), _bf16_bits(fresh)
    assert np.array_equal(oracle.bf16_decode(fb), fresh)
    idx = np.array([[1, 5, 8, 13, 21]])
    out, mu_hat = oracle.mean_correct(rb, fb, [0], 1, 1e4, False, idx, np.ones((1, n)))
    e = mu_hat - mu
    np.testing.assert_allclose(e, xi[:, :, idx[0]].mean(axis=2), atol=1e-15)
    got = oracle.bf16_decode(out) - fresh
    want = e[:, :, None] - xi
    mask = np.ones(n, bool)
    mask[idx[0]] = False
    exact = reuse + mu_hat[:, :, None]                # the value before bf16 rounding
    half_ulp = 2.0 ** -8 * np.abs(exact)              # half a bf16 ulp, relative
    assert np.all(np.abs(got - want)[:, :, mask] <= half_ulp[:, :, mask])


# ------------------------------------------------------------------ low rank

def test_lowrank_zero_factor_is_identity():
    rng = np.random.default_rng(13)
    C, L, n, H, D, r = 1, 2, 9, 2, 16, 4
    x = _bf16_bits(rng.standard_normal((C, L, n, H, D)))
    A = np.zeros((C, L, H, n, r), np.uint16)
    B = _bf16_bits(rng.standard_normal((C, L, H, r, D)))
    assert np.array_equal(oracle.lowrank_apply(x, A, B), x)


def test_lowrank_one_hot_rows_pick_b_rows():
    rng = np.random.default_rng(14)
    C, L, n, H, D, r = 1, 1, 6, 2, 8, 3
    x = _bf16_bits(rng.standard_normal((C, L, n, H, D)))
    A = np.zeros((C, L, H, n, r))
    pick = rng.integers(0, r, (H, n))
    for h in range(H):
        for j in range(n):
            A[0, 0, h, j, pick[h, j]] = 1.0
    Bd = rng.standard_normal((C, L, H, r, D))
    out = oracle.lowrank_apply(x, _bf16_bits(A), _bf16_bits(Bd))
    Bq = oracle.bf16_decode(_bf16_bits(Bd))
    xd = oracle.bf16_decode(x)
    for h in range(H):
        for j in range(n):
            assert np.array_equal(out[0, 0, j, h], _bf16_bits(xd[0, 0, j, h] + Bq[0, 0, h, pick[h, j]]))


def test_lowrank_matches_numpy_matmul():
    rng = np.random.default_rng(15)
    C, L, n, H, D, r = 2, 2, 33, 3, 16, 16
    x = _bf16_bits(rng.standard_normal((C, L, n, H, D)))
    A = _bf16_bits(0.1 * rng.standard_normal((C, L, H, n, r)))
    B = _bf16_bits(rng.standard_normal((C, L, H, r, D)))
    out = oracle.lowrank_apply(x, A, B)
    delta = np.matmul(oracle.bf16_decode(A), oracle.bf16_decode(B))  # [C][L][H][n][D]
    ref = oracle.bf16_decode(x) + np.transpose(delta, (0, 1, 3, 2, 4))
    got = oracle.bf16_decode(out)
    # same value up to summation order; bf16 rounding can differ only at exact boundaries
    assert np.mean(out == _bf16_bits(ref)) > 0.999
    np.testing.assert_allclose(got, ref, rtol=2.0 ** -8, atol=1e-6)


# ------------------------------------------------------------------ draft rank

def _draft_case(rng, C=1, L=3, n=40, Hkv=2, Hq=4, D=16, T=2, scale=1.0):
    k = _bf16_bits(scale * rng.standard_normal((C, L, n, Hkv, D)))
    q = _bf16_bits(rng.standard_normal((C, L, T, Hq, D)))
    return k, q


def test_draft_scores_sum_to_query_count():
    rng = np.random.default_rng(16)
    k, q = _draft_case(rng, C=2, L=4)
    a = oracle.draft_scores(k, q, layer_begin=1)
    np.testing.assert_allclose(a.sum(axis=1), (4 - 1) * 2 * 4, rtol=1e-12)
    assert np.all(a > 0)


def test_draft_scores_common_key_shift_invariance():
    """Adding one vector to every key of a (layer, head) adds one constant to every
    logit, which softmax cancels (AgentKVShift, limitations: common key shift)."""
    rng = np.random.default_rng(17)
    C, L, n, Hkv, D = 1, 3, 24, 2, 8
    kd = rng.integers(-8, 8, (C, L, n, Hkv, D)) / 8.0
    qd = rng.integers(-8, 8, (C, L, 2, 4, D)) / 8.0
    shift = rng.integers(-8, 8, (C, L, 1, Hkv, D)) / 4.0
    a0 = oracle.draft_scores(_bf16_bits(kd), _bf16_bits(qd), 1)
    a1 = oracle.draft_scores(_bf16_bits(kd + shift), _bf16_bits(qd), 1)
    np.testing.assert_allclose(a1, a0, rtol=1e-11, atol=1e-13)


def test_draft_scores_matches_library_softmax():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(18)
    C, L, n, Hkv, Hq, D, T = 1, 3, 50, 2, 6, 8, 2
    k, q = _draft_case(rng, C, L, n, Hkv, Hq, D, T)
    a = oracle.draft_scores(k, q, 1)
    kd, qd = oracle.bf16_decode(k), oracle.bf16_decode(q)
    ref = np.zeros(n)
    for l in range(1, L):
        for t in range(T):
            for h in range(Hq):
                z = kd[0, l, :, h // (Hq // Hkv)] @ qd[0, l, t, h] / math.sqrt(D)
                ref += sp.softmax(z)
    np.testing.assert_allclose(a[0], ref, rtol=1e-12)


def test_draft_identical_keys_and_dominant_key():
    rng = np.random.default_rng(19)
    C, L, n, Hkv, Hq, D = 1, 2, 30, 1, 2, 8
    row = rng.standard_normal(D)
    k = _bf16_bits(np.broadcast_to(row, (C, L, n, Hkv, D)).copy())
    q = _bf16_bits(rng.standard_normal((C, L, 2, Hq, D)))
    a = oracle.draft_scores(k, q, 1)[0]
    assert np.allclose(a, a[0], rtol=1e-14)
    assert list(oracle.topk(a, 5, False)) == [0, 1, 2, 3, 4]
    kd = rng.standard_normal((C, L, n, Hkv, D)) * 0.01
    qd = np.ones((C, L, 2, Hq, D))
    kd[0, :, 17, 0, :] = 4.0
    a = oracle.draft_scores(_bf16_bits(kd), _bf16_bits(qd), 1)[0]
    assert list(oracle.topk(a, 1, False)) == [17]
    assert a[17] > 0.999 * (L - 1) * 2 * Hq


def test_softmax_counterexample_l1():
    """Two keys with logits (z, -z): the softmax mass on key 0 is (1 + tanh z)/2, so the
    L1 distance from the uniform pair is tanh z; at z = 0.1 the page prints 0.099668."""
    g = _golden("softmax_l1_counterexample.txt")
    assert abs(math.tanh(g["logits_b"][0]) - g["l1_distance"][0]) < 0.5e-6
    # one layer scored, one step, one head, D = 1: the logit is q * k exactly
    kd = np.zeros((1, 2, 2, 1, 1))                    # [C][L][n][H][D]
    kd[0, :, 0] = 0.2
    kd[0, :, 1] = -0.2
    kb = _bf16_bits(kd)
    q = _bf16_bits(np.full((1, 2, 1, 1, 1), 0.5))
    z = 0.5 * oracle.bf16_decode(kb)[0, 1, 0, 0, 0]
    a = oracle.draft_scores(kb, q, 1)[0]
    l1 = abs(a[0] - 0.5) + abs(a[1] - 0.5)
    assert abs(l1 - math.tanh(z)) < 1e-14
    assert abs(l1 - g["l1_distance"][0]) < 2e-4


def test_row_overwrite_all_rows_is_fresh():
    rng = np.random.default_rng(20)
    kv = _bf16_bits(rng.standard_normal((2, 3, 10, 2, 8)))
    fresh = _bf16_bits(rng.standard_normal((2, 3, 10, 2, 8)))
    idx = np.tile(np.arange(10), (2, 1))
    assert np.array_equal(oracle.row_overwrite(kv, fresh, idx), fresh)
    part = oracle.row_overwrite(kv, fresh, np.array([[2, 7], [0, 9]]))
    assert np.array_equal(part[0, :, 2], fresh[0, :, 2]) and np.array_equal(part[0, :, 3], kv[0, :, 3])


# ---------------------------------------------------------- diff encode/gather

def _siblings(rng, S=4, L=2, n=64, H=2, D=8, bt=16, frac=0.3):
    mk = _bf16_bits(rng.standard_normal((L, n, H, D)))
    mv = _bf16_bits(rng.standard_normal((L, n, H, D)))
    sk = np.repeat(mk[None], S, 0)
    sv = np.repeat(mv[None], S, 0)
    for s in range(S):
        for l in range(L):
            for blk in range(n // bt):
                if rng.random() < frac:
                    plane = sk if rng.random() < 0.5 else sv
                    t = blk * bt + int(rng.integers(0, bt))
                    plane[s, l, t, int(rng.integers(0, H)), int(rng.integers(0, D))] ^= 1
    return mk, mv, sk, sv


def test_diff_roundtrip_and_counts():
    rng = np.random.default_rng(21)
    mk, mv, sk, sv = _siblings(rng)
    mask, offs, payload, total = oracle.diff_encode(mk, mv, sk, sv, 16)
    bits = np.unpackbits(mask.view(np.uint8), bitorder="little")[: offs.size - 1]
    assert total == int(bits.sum()) == offs[-1]
    assert np.array_equal(offs[:-1], np.concatenate([[0], np.cumsum(bits)[:-1]]))
    ok, ov = oracle.diff_gather(mk, mv, mask, offs, payload, sk.shape[0], 16)
    assert np.array_equal(ok, sk) and np.array_equal(ov, sv)


def test_diff_identical_and_all_different():
    rng = np.random.default_rng(22)
    mk, mv, _, _ = _siblings(rng, frac=0)
    S = 3
    same_k, same_v = np.repeat(mk[None], S, 0), np.repeat(mv[None], S, 0)
    mask, offs, payload, total = oracle.diff_encode(mk, mv, same_k, same_v, 16)
    assert total == 0 and not mask.any() and not offs.any()
    dk, dv = same_k ^ 1, same_v.copy()
    mask, offs, payload, total = oracle.diff_encode(mk, mv, dk, dv, 16)
    L, n, H, D = mk.shape
    assert total == S * L * (n // 16)
    blocks = dk.reshape(S, L, n // 16, 16, H, D).reshape(-1, 16, H, D)
    assert np.array_equal(payload[:, 0], blocks)
    assert np.array_equal(payload[:, 1], dv.reshape(-1, 16, H, D))


def test_diff_is_bitwise_signed_zero():
    """+0 and -0 compare equal as numbers but are different bf16 words: the block is dirty."""
    L, n, H, D = 1, 32, 1, 8
    mk = np.zeros((L, n, H, D), np.uint16)
    mv = np.zeros_like(mk)
    sk = mk[None].copy()
    sk[0, 0, 20, 0, 3] = 0x8000
    mask, offs, payload, total = oracle.diff_encode(mk, mv, sk, mv[None].copy(), 16)
    assert total == 1 and mask[0] == 0b10


def test_diff_capacity_reports_need():
    rng = np.random.default_rng(23)
    mk, mv, sk, sv = _siblings(rng, frac=0.5)
    _, offs, _, total = oracle.diff_encode(mk, mv, sk, sv, 16)
    _, offs2, payload, total2 = oracle.diff_encode(mk, mv, sk, sv, 16, capacity_entries=total - 1)
    assert total2 == total and np.array_equal(offs, offs2)


# ------------------------------------------------------------ fused diff restore

def _restore_case(rng, S=3, L=2, n=64, H=2, D=16, bt=16, slots=250, skip=0.1):
    mk, mv, sk, sv = _siblings(rng, S=S, L=L, n=n, H=H, D=D, bt=bt, frac=0.5)
    mask, offs, payload, _ = oracle.diff_encode(mk, mv, sk, sv, bt)
    slot_map = rng.permutation(slots)[: S * n].reshape(S, n).astype(np.int32)
    slot_map[rng.random((S, n)) < skip] = -1
    slot_map[0, 1] = slots          # past the pool: not restored either
    pool = np.full((L, slots, H, D), 0x1234, np.uint16)
    return mk, mv, sk, sv, mask, offs, payload, slot_map, pool


def test_diff_restore_zero_shift_places_each_mirror_row():
    """Zero shift: pool row slot_map[s][t] of layer l holds mirror s's token t bit for bit
    (keys and values); skipped and unmapped rows keep their contents."""
    rng = np.random.default_rng(31)
    mk, mv, sk, sv, mask, offs, payload, smap, pool = _restore_case(rng)
    S, L, n = sk.shape[:3]
    pk, pv = oracle.diff_restore(mk, mv, mask, offs, payload, S, 16, np.zeros(S), 1e4, smap, pool, pool)
    hit = np.zeros(pool.shape[1], bool)
    for s in range(S):
        for t in range(n):
            slot = smap[s, t]
            if 0 <= slot < pool.shape[1]:
                hit[slot] = True
                assert np.array_equal(pk[:, slot], sk[s, :, t]) and np.array_equal(pv[:, slot], sv[s, :, t])
    assert (pk[:, ~hit] == 0x1234).all() and (pv[:, ~hit] == 0x1234).all()
    assert hit.sum() < S * n        # some tokens were skipped


def test_diff_restore_rotates_keys_by_the_mirror_shift():
    """Keys of mirror s are rotated by delta[s] (complex multiplication by exp(i delta theta)),
    values are copied unrotated."""
    rng = np.random.default_rng(32)
    mk, mv, sk, sv, mask, offs, payload, smap, pool = _restore_case(rng, skip=0.0)
    S, L, n, H, D = sk.shape
    delta = np.array([0, 137, -4000], np.int32)
    base = 5e5
    pk, pv = oracle.diff_restore(mk, mv, mask, offs, payload, S, 16, delta, base, smap, pool, pool)
    rot = oracle.rerope(sk, delta, base)
    th = np.power(base, -2.0 * np.arange(D // 2) / D)
    for s in range(S):
        ok = smap[s] < pool.shape[1]
        got_k = pk[:, smap[s, ok]]
        assert np.array_equal(got_k, rot[s][:, ok])
        assert np.array_equal(pv[:, smap[s, ok]], sv[s][:, ok])
        x = oracle.bf16_decode(sk[s][:, ok])
        z = (x[..., : D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * float(delta[s]) * th)
        y = oracle.bf16_decode(got_k)
        tol = np.abs(np.concatenate([z.real, z.imag], -1)) * 2.0 ** -8 + 1e-30
        assert (np.abs(y - np.concatenate([z.real, z.imag], -1)) <= tol).all()


# ------------------------------------------------------------ anchor-pool correction

def _anchor_case(rng, C=2, V=3, L=2, n=7, F=16, r=4, a_std=0.5):
    x = _bf16_bits(rng.standard_normal((C, L, n, F)))
    a = _bf16_bits(a_std * rng.standard_normal((C, V, L, n, r)))
    b = _bf16_bits(rng.standard_normal((C, V, L, F, r)))
    return x, a, b


def _recon(a, b):
    """numpy: A [.., n, r] @ B^T for b stored [.., F, r]."""
    return np.matmul(oracle.bf16_decode(a), np.swapaxes(oracle.bf16_decode(b), -1, -2))


def test_anchor_gate_matches_frobenius_softmax_and_entropy():
    """d_v against numpy's Frobenius norm of the prefix residual over layers, g against
    scipy's softmax, the normalised entropy against scipy's entropy in bits."""
    from scipy.special import softmax
    from scipy.stats import entropy
    rng = np.random.default_rng(41)
    x, a, b = _anchor_case(rng, a_std=0.05)
    k = 5
    d, g, hbar, acc = oracle.anchor_gate(x, a, b, k, T=1.0, tau=0.6)
    C, V = d.shape
    for c in range(C):
        res = oracle.bf16_decode(x[c])[None, :, :k] - _recon(a[c], b[c])[:, :, :k]  # [V][L][k][F]
        dn = np.linalg.norm(res.reshape(V, -1), axis=1)
        np.testing.assert_allclose(d[c], dn, rtol=1e-12)
        np.testing.assert_allclose(g[c], softmax(-dn), rtol=1e-10)
        h = entropy(g[c], base=2) / np.log2(V)
        assert abs(hbar[c] - h) < 1e-12 and acc[c] == (h <= 0.6)


def test_anchor_gate_special_cases():
    rng = np.random.default_rng(42)
    x, a, b = _anchor_case(rng, C=1, V=4)
    same_a, same_b = np.repeat(a[:, :1], 4, 1), np.repeat(b[:, :1], 4, 1)
    d, g, hbar, acc = oracle.anchor_gate(x, same_a, same_b, 3, tau=0.999)
    assert np.all(g == 0.25) and abs(hbar[0] - 1.0) < 1e-15 and not acc[0]     # flat: no reuse
    assert oracle.anchor_gate(x, same_a, same_b, 3, tau=1.0)[3][0]
    d, g, hbar, acc = oracle.anchor_gate(x, a[:, :1], b[:, :1], 3, tau=1.0)
    assert np.isnan(hbar[0]) and not acc[0]                                    # one anchor: dense
    # two anchors on x = 0 reconstructing 0 and the constant e: d = (0, |e| sqrt(L k F)),
    # g = (1, exp(-d1)) / (1 + exp(-d1)), Hbar = the binary entropy of g_0 (log2 2 = 1)
    L, n, F, k = 1, 1, 1, 1
    x0 = np.zeros((1, L, n, F), np.uint16)
    aa = _bf16_bits(np.array([0.0, 1.0]).reshape(1, 2, 1, 1, 1))
    bb = _bf16_bits(np.array([1.0, np.log(3.0)]).reshape(1, 2, 1, 1, 1))
    d, g, hbar, acc = oracle.anchor_gate(x0, aa, bb, k, tau=0.9)
    e = float(oracle.bf16_decode(bb)[0, 1, 0, 0, 0])
    g0 = 1.0 / (1.0 + math.exp(-e))
    assert d[0, 0] == 0.0 and d[0, 1] == e
    assert abs(g[0, 0] - g0) < 1e-15
    hb = -(g0 * math.log2(g0) + (1 - g0) * math.log2(1 - g0))
    assert abs(hbar[0] - hb) < 1e-12 and acc[0] == (hb <= 0.9)
    # a far anchor set against one exact match: the distribution is one-hot, entropy 0
    xs = _bf16_bits(np.full((1, 1, 2, 4), 2.0))
    a3 = _bf16_bits(np.array([1.0, 40.0, -40.0]).reshape(1, 3, 1, 1, 1).repeat(2, 3))
    b3 = _bf16_bits(np.full((1, 3, 1, 4, 1), 2.0))
    d, g, hbar, acc = oracle.anchor_gate(xs, a3, b3, 2, tau=0.01)
    assert d[0, 0] == 0.0 and g[0, 0] == 1.0 and hbar[0] < 1e-80 and acc[0]


def test_anchor_weights_match_library_softmax():
    """w = softmax(-mean|x - A B|) per token, against numpy + scipy; one anchor -> 1,
    identical anchors -> 1/V."""
    from scipy.special import softmax
    rng = np.random.default_rng(43)
    x, a, b = _anchor_case(rng, C=2, V=4, n=9, F=32, r=8)
    w = oracle.anchor_weights(x, a, b)
    for c in range(2):
        m = np.abs(oracle.bf16_decode(x[c])[None] - _recon(a[c], b[c])).mean(-1)  # [V][L][n]
        ref = softmax(-np.moveaxis(m, 0, -1), axis=-1)
        np.testing.assert_allclose(w[c], ref, rtol=1e-12)
    assert np.all(oracle.anchor_weights(x, a[:, :1], b[:, :1]) == 1.0)
    w4 = oracle.anchor_weights(x, np.repeat(a[:, :1], 4, 1), np.repeat(b[:, :1], 4, 1))
    assert np.all(w4 == 0.25)


def test_anchor_correct_special_cases():
    """Zero deltas give the aligned source (rerope for keys, the source for values) bit
    for bit; one anchor of weight 1 without alignment is x + A B, against numpy."""
    rng = np.random.default_rng(44)
    C, V, L, n, H, D, r = 2, 3, 2, 6, 2, 16, 4
    x = _bf16_bits(rng.standard_normal((C, L, n, H * D)))
    ad = np.zeros((C, V, L, n, r), np.uint16)
    bd = _bf16_bits(rng.standard_normal((C, V, L, H * D, r)))
    w = rng.dirichlet(np.ones(V), (C, L, n))
    delta = np.array([300, -7])
    out = oracle.anchor_correct(x, ad, bd, w, H, delta, 1e4, rotate=True)
    assert np.array_equal(out, oracle.rerope(x.reshape(C, L, n, H, D), delta, 1e4).reshape(x.shape))
    assert np.array_equal(oracle.anchor_correct(x, ad, bd, w, H, delta, 1e4, rotate=False), x)
    a1 = _bf16_bits(0.3 * rng.standard_normal((C, 1, L, n, r)))
    out = oracle.anchor_correct(x, a1, bd[:, :1], np.ones((C, L, n, 1)), H, delta, 1e4, rotate=False)
    ref = oracle.bf16_decode(x) + _recon(a1, bd[:, :1])[:, 0]
    assert np.mean(out == _bf16_bits(ref)) > 0.999
    np.testing.assert_allclose(oracle.bf16_decode(out), ref, rtol=2.0 ** -8, atol=1e-6)


def test_anchor_correct_is_weighted_sum_of_anchor_deltas():
    """Weights put the anchors' deltas together linearly: against the numpy sum of
    w_v (A_v B_v) added to the rotated source."""
    rng = np.random.default_rng(45)
    C, V, L, n, H, D, r = 1, 4, 2, 5, 2, 16, 8
    x = _bf16_bits(rng.standard_normal((C, L, n, H * D)))
    ad = _bf16_bits(0.2 * rng.standard_normal((C, V, L, n, r)))
    bd = _bf16_bits(rng.standard_normal((C, V, L, H * D, r)))
    w = rng.dirichlet(np.ones(V), (C, L, n))
    out = oracle.anchor_correct(x, ad, bd, w, H, [55], 5e5, rotate=True)
    rot = oracle.rotate_f64(oracle.bf16_decode(x).reshape(C, L, n, H, D), 55, 5e5).reshape(x.shape)
    ref = rot + np.einsum("clnv,cvlnf->clnf", w, _recon(ad, bd))
    np.testing.assert_allclose(oracle.bf16_decode(out), ref, rtol=2.0 ** -8, atol=1e-6)


def test_anchor_order_does_not_matter():
    """Relabelling the anchors permutes d, g and the weights the same way and leaves the
    entropy, the verdict and (up to the order of a double sum) the correction unchanged:
    catches an anchor index crossed between A and B or between weights and deltas."""
    rng = np.random.default_rng(46)
    C, V, L, n, H, D, r = 2, 5, 2, 6, 2, 16, 4
    x, a, b = _anchor_case(rng, C=C, V=V, L=L, n=n, F=H * D, r=r, a_std=0.3)
    ad = _bf16_bits(0.2 * rng.standard_normal((C, V, L, n, r)))
    bd = _bf16_bits(rng.standard_normal((C, V, L, H * D, r)))
    perm = np.array([3, 0, 4, 1, 2])
    d, g, hbar, acc = oracle.anchor_gate(x, a, b, 4, tau=0.7)
    dp, gp, hp, ap = oracle.anchor_gate(x, a[:, perm], b[:, perm], 4, tau=0.7)
    np.testing.assert_array_equal(dp, d[:, perm])
    np.testing.assert_allclose(gp, g[:, perm], rtol=1e-14)
    np.testing.assert_allclose(hp, hbar, rtol=1e-13)
    assert np.array_equal(ap, acc)
    w = oracle.anchor_weights(x, a, b)
    wp = oracle.anchor_weights(x, a[:, perm], b[:, perm])
    np.testing.assert_allclose(wp, w[..., perm], rtol=1e-14)
    out = oracle.anchor_correct(x, ad, bd, w, H, [9, 400], 1e4, rotate=True)
    outp = oracle.anchor_correct(x, ad[:, perm], bd[:, perm], wp, H, [9, 400], 1e4, rotate=True)
    assert np.mean(out == outp) > 0.999
    np.testing.assert_allclose(oracle.bf16_decode(outp), oracle.bf16_decode(out), rtol=2.0 ** -8, atol=1e-6)


# ------------------------------------------------------------ repair layouts

def test_chunk_budgets_reproduce_table8():
    """The chunk budget max(1, round(rho n / B)) reproduces every printed budget of the
    unit-of-choice table (no skip rule there: the whole-segment row is a single chunk)."""
    rows = _golden("bcr_table8_budgets.txt")
    rng = np.random.default_rng(51)
    s = rng.random((1, 2048))
    for key, (unit, pct) in rows.items():
        _, counts = oracle.repair_layout(s, oracle.LAYOUT_CHUNK, chunk_tokens=int(unit), budget=(1, 5), skip=False)
        assert round(100.0 * counts[0] / 2048, 1) == pct, key


def test_chunk_skip_rule_and_short_last_chunk():
    rng = np.random.default_rng(52)
    s = rng.random((1, 200))
    assert oracle.repair_layout(s, oracle.LAYOUT_CHUNK, 128, (1, 5))[1][0] == 0       # n < 2B
    assert oracle.repair_layout(s, oracle.LAYOUT_CHUNK, 64, (1, 5))[1][0] == 0        # rho n < B
    means = [s[0, a:a + 64].mean() for a in (0, 64, 128, 192)]
    best = int(np.argmax(means))
    assert oracle.repair_layout(s, oracle.LAYOUT_CHUNK, 64, (1, 3))[1][0] == (8 if best == 3 else 64)
    # a short last chunk is scored by its own mean: make it the best
    s2 = np.zeros((1, 200))
    s2[0, 192:] = 1.0
    s2[0, :64] = 0.9
    idx, cnt = oracle.repair_layout(s2, oracle.LAYOUT_CHUNK, 64, (1, 2))
    assert cnt[0] == 64 + 8 and list(idx[0, :cnt[0]]) == list(range(64)) + list(range(192, 200))


def test_chunk_layout_is_best_subset_by_brute_force():
    """Top chunks by mean = the chunk subset of the budget's size with the largest sum of
    means (distinct means), found by enumeration."""
    rng = np.random.default_rng(53)
    for trial in range(20):
        n, B = int(rng.integers(12, 40)), int(rng.integers(2, 7))
        s = rng.random((1, n))
        idx, cnt = oracle.repair_layout(s, oracle.LAYOUT_CHUNK, B, (1, 3), skip=False)
        nch = (n + B - 1) // B
        means = [s[0, i * B:min(n, i * B + B)].mean() for i in range(nch)]
        c = max(1, int(round(n / (3 * B))))
        c = min(c, nch)
        best = max(itertools.combinations(range(nch), c), key=lambda sub: sum(means[i] for i in sub))
        rows = sorted(j for i in best for j in range(i * B, min(n, i * B + B)))
        assert list(idx[0, :cnt[0]]) == rows


def test_single_layout_matches_lexsort():
    rng = np.random.default_rng(54)
    s = np.round(rng.random((3, 500)) * 50) / 50            # many ties
    idx, cnt = oracle.repair_layout(s, oracle.LAYOUT_SINGLE, budget=(1, 10))
    for u in range(3):
        top = np.lexsort((np.arange(500), -s[u]))[:50]
        assert cnt[u] == 50 and list(idx[u, :50]) == sorted(top)


def _spans(rows):
    rows = sorted(rows)
    out, start = [], rows[0]
    for a, b in zip(rows, rows[1:] + [None]):
        if b != a + 1:
            out.append((start, a))
            start = b
    return out


def test_grow_layout_invariants_and_limits():
    rng = np.random.default_rng(55)
    n = 400
    s = rng.random((2, n)) ** 3
    k = 80
    # tau > 1: nothing grows, the single layout
    g, cg = oracle.repair_layout(s, oracle.LAYOUT_GROW, budget=(1, 5), tau=1.5)
    t, ct = oracle.repair_layout(s, oracle.LAYOUT_SINGLE, budget=(1, 5))
    assert np.array_equal(g, t) and np.array_equal(cg, ct)
    # tau = 0: one span of k rows around the best row
    g, cg = oracle.repair_layout(s, oracle.LAYOUT_GROW, budget=(1, 5), tau=0.0)
    for u in range(2):
        rows = list(g[u, :cg[u]])
        assert cg[u] == k and _spans(rows) == [(rows[0], rows[-1])] and int(np.argmax(s[u])) in rows
    # tau = 0.25: exactly k distinct rows, the best row among them, fewer spans than with
    # no growth at all and more than with unlimited growth
    g, cg = oracle.repair_layout(s, oracle.LAYOUT_GROW, budget=(1, 5), tau=0.25)
    for u in range(2):
        rows = list(g[u, :cg[u]])
        assert cg[u] == k and len(set(rows)) == k and int(np.argmax(s[u])) in rows
        assert 1 < len(_spans(rows)) < len(_spans(list(t[u, :ct[u]])))


def test_grow_layout_small_case_by_hand():
    """A worked case: scores 1 5 4 0.9 0.1 8 7 0.5, budget 4 of 8 rows (rho 1/2), tau 0.5.
    Seed 5 (8): left 0.1 < 4, right 6 (7) >= 4 -> {5,6}; then 7 (0.5) < 4, 4 (0.1) < 4:
    span ends.  Next seed 1 (5): neighbours 0 (1) < 2.5, 2 (4) >= 2.5 -> {1,2}: budget
    spent.  Rows 1 2 5 6."""
    s = np.array([[1, 5, 4, 0.9, 0.1, 8, 7, 0.5]], dtype=np.float64)
    idx, cnt = oracle.repair_layout(s, oracle.LAYOUT_GROW, budget=(1, 2), tau=0.5)
    assert cnt[0] == 4 and list(idx[0, :4]) == [1, 2, 5, 6]


# ------------------------------------------------------------ master selection, split diffs

def test_master_select_matches_numpy():
    rng = np.random.default_rng(61)
    A, R, n = 5, 3, 70
    dk = rng.random((A * R, n)).astype(np.float32)
    dv = rng.random((A * R, n)).astype(np.float32)
    m, tot = oracle.master_select(dk, dv, A)
    ref = dk.astype(np.float64).reshape(A, -1).sum(1) + dv.astype(np.float64).reshape(A, -1).sum(1)
    np.testing.assert_allclose(tot, ref, rtol=1e-12)
    assert m == int(np.argmin(ref))
    m1, tot1 = oracle.master_select(dk, None, A)
    np.testing.assert_allclose(tot1, dk.astype(np.float64).reshape(A, -1).sum(1), rtol=1e-12)
    same = np.tile(dk[:R], (A, 1))
    assert oracle.master_select(same, same, A)[0] == 0          # ties to the lower index


def test_master_by_deviation_minimises_diff_storage():
    """Agents share content X and each changes a disjoint set of its blocks; the agent with
    the smallest total deviation from X is the master whose diffs of the others take the
    fewest payload entries (entries(m) = sum |M| + (S - 2) |M_m|)."""
    rng = np.random.default_rng(62)
    S, L, n, H, D, bt = 5, 2, 64, 2, 8, 8
    X_k = _bf16_bits(rng.standard_normal((L, n, H, D)))
    X_v = _bf16_bits(rng.standard_normal((L, n, H, D)))
    nblk = n // bt
    blocks = rng.permutation(L * nblk)
    sizes = [3, 1, 4, 2, 5]
    caches_k = np.repeat(X_k[None], S, 0)
    caches_v = np.repeat(X_v[None], S, 0)
    start = 0
    for s in range(S):
        for b in blocks[start:start + sizes[s]]:
            l, blk = divmod(int(b), nblk)
            noise = rng.standard_normal((bt, H, D))
            caches_k[s, l, blk * bt:(blk + 1) * bt] = _bf16_bits(oracle.bf16_decode(X_k[l, blk * bt:(blk + 1) * bt]) + noise)
        start += sizes[s]
    dev = np.sqrt(((oracle.bf16_decode(caches_k) - oracle.bf16_decode(X_k)[None]) ** 2).sum(axis=(3, 4)))
    d = dev.reshape(S * L, n).astype(np.float32)                     # [agent * layer][token]
    m, _ = oracle.master_select(d, None, S)
    entries = []
    for cand in range(S):
        _, _, _, total = oracle.diff_encode(caches_k[cand], caches_v[cand], caches_k, caches_v, bt)
        entries.append(total)
    assert m == int(np.argmin(entries)) == 1


def _split_case(rng, S=3, L=2, n=48, H=2, D=8, bt=8):
    mk = _bf16_bits(rng.standard_normal((L, n, H, D)))
    mv = _bf16_bits(rng.standard_normal((L, n, H, D)))
    sk = np.repeat(mk[None], S, 0)
    sv = np.repeat(mv[None], S, 0)
    return mk, mv, sk, sv, bt


def test_split_diff_roundtrip_and_relation_to_joint():
    rng = np.random.default_rng(63)
    mk, mv, sk, sv, bt = _split_case(rng)
    S, L, n = sk.shape[:3]
    for s in range(S):
        for l in range(L):
            for blk in range(n // bt):
                u = rng.random()
                t = blk * bt + int(rng.integers(0, bt))
                if u < 0.2:
                    sk[s, l, t, 0, 0] ^= 1
                elif u < 0.4:
                    sv[s, l, t, 1, 3] ^= 1
                elif u < 0.5:
                    sk[s, l, t, 1, 1] ^= 1
                    sv[s, l, t, 0, 2] ^= 1
    kd, vd = oracle.diff_encode_split(mk, mv, sk, sv, bt)
    ok, ov = oracle.diff_gather_split(mk, mv, kd, vd, S, bt)
    assert np.array_equal(ok, sk) and np.array_equal(ov, sv)
    jmask, joffs, jpay, jtotal = oracle.diff_encode(mk, mv, sk, sv, bt)
    assert np.array_equal(kd[0] | vd[0], jmask)                     # joint dirty = K dirty or V dirty
    nk, nv = int(kd[1][-1]), int(vd[1][-1])
    assert max(nk, nv) <= jtotal <= nk + nv and nk + nv > jtotal    # some blocks touch one plane only


def test_split_diff_equals_joint_when_planes_agree():
    """When K and V touch the same blocks the two lists coincide with the joint one and the
    split payloads are the joint payload's K and V halves."""
    rng = np.random.default_rng(64)
    mk, mv, sk, sv, bt = _split_case(rng)
    for s, l, t in ((0, 0, 3), (1, 1, 40), (2, 0, 17), (2, 1, 9)):
        sk[s, l, t, 0, 0] ^= 2
        sv[s, l, t, 1, 1] ^= 2
    kd, vd = oracle.diff_encode_split(mk, mv, sk, sv, bt)
    jmask, joffs, jpay, jtotal = oracle.diff_encode(mk, mv, sk, sv, bt)
    assert np.array_equal(kd[0], jmask) and np.array_equal(vd[0], jmask)
    assert np.array_equal(kd[1], joffs) and np.array_equal(vd[1], joffs)
    assert np.array_equal(kd[2], jpay[:, 0]) and np.array_equal(vd[2], jpay[:, 1])
