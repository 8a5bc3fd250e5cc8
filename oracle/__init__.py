"""CPU oracle for the reused-KV-chunk repair path.

TEST INFRASTRUCTURE: only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package.  The product (the CUDA library
and its Python binding) never imports it, and the two share no code.

The arithmetic lives in ``kvfix_oracle.c`` (plain C, double precision, one loop nest
per definition, each citing the passage it follows).  This module only builds that
file with gcc and marshals numpy arrays into it.  bf16 tensors travel as ``uint16``
arrays holding the raw bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvfix_oracle.c")
_LIB = os.path.join(_HERE, "libkvfix_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, OpenMP) if stale."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(
                ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
                 "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        D = ctypes.c_double
        sig = {
            "oracle_bf16_encode": (None, [P, P, I64]),
            "oracle_bf16_decode": (None, [P, P, I64]),
            "oracle_num_threads": (I, []),
            "oracle_set_num_threads": (None, [I]),
            "oracle_rope_theta": (None, [D, I, P]),
            "oracle_rotate_f64": (None, [P, P, I64, I, D, D]),
            "oracle_rerope": (None, [P, P, I, I, I, I, I, P, D]),
            "oracle_compose_fresh": (None, [P, P, P, P, I, I, I, I, I, I, D, I, P]),
            "oracle_scores": (None, [P, P, I, I, I, I, I, P, D, I, P]),
            "oracle_topk": (None, [P, I, I, I, P]),
            "oracle_mean_correct": (None, [P, P, I, I, I, I, I, I, P, D, I, P, I, P, P, P]),
            "oracle_correct_with_weights": (D, [P, I, P, P, I, P]),
            "oracle_lowrank_apply": (None, [P, P, P, I, I, I, I, I, I, P]),
            "oracle_draft_scores": (None, [P, P, I, I, I, I, I, I, I, I, P]),
            "oracle_row_overwrite": (None, [P, P, I, I, I, I, I, P, I]),
            "oracle_diff_encode": (I64, [P, P, P, P, I, I, I, I, I, I, P, P, P, I64]),
            "oracle_diff_gather": (None, [P, P, P, P, P, I, I, I, I, I, I, P, P]),
            "oracle_diff_restore": (None, [P, P, P, P, P, I, I, I, I, I, I, P, D, P, I64, P, P]),
            "oracle_anchor_gate": (None, [P, P, P, I, I, I, I, I, I, I, D, D, P, P, P, P]),
            "oracle_repair_layout": (I, [P, I, I, I, I, I, I, D, I, P, I, P]),
            "oracle_master_select": (I, [P, P, I, I, I, P]),
            "oracle_diff_encode_split": (None, [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, P]),
            "oracle_diff_gather_split": (None, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P]),
            "oracle_anchor_weights": (None, [P, P, P, I, I, I, I, I, I, D, P]),
            "oracle_anchor_correct": (None, [P, P, P, P, I, I, I, I, I, I, I, P, D, I, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"bf16 arrays travel as uint16 bit patterns, got {a.dtype}"
    return a


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# ----------------------------------------------------------------- bf16

def bf16_encode(x) -> np.ndarray:
    """double -> float (nearest even) -> bf16 (nearest even), as uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_bf16_encode(_p(x), _p(out), x.size)
    return out


def bf16_decode(h) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, np.float64)
    _load().oracle_bf16_decode(_p(h), _p(out), h.size)
    return out


# ----------------------------------------------------------------- RoPE

def rope_theta(base: float, D: int) -> np.ndarray:
    out = np.empty(D // 2, np.float64)
    _load().oracle_rope_theta(float(base), int(D), _p(out))
    return out


def rotate_f64(x, delta: float, base: float) -> np.ndarray:
    """Rotate double rows (last axis = head_dim) by delta positions, no rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    D = x.shape[-1]
    y = np.empty_like(x)
    _load().oracle_rotate_f64(_p(x), _p(y), x.size // D, D, float(delta), float(base))
    return y


def rerope(k, delta, base: float) -> np.ndarray:
    """k: [C][L][n][H][D] uint16; delta: [C] int."""
    k = _u16(k)
    C, L, n, H, D = k.shape
    d = np.ascontiguousarray(delta, dtype=np.int32).reshape(C)
    out = np.empty_like(k)
    _load().oracle_rerope(_p(k), _p(out), C, L, n, H, D, _p(d), float(base))
    return out


def compose_fresh(reuse, mu, xi, delta, agents: int, base: float, rotate_keys: bool) -> np.ndarray:
    """Synthetic fresh states: bf16(rot(reuse) + mu + xi).

    reuse [R][L][n][H][D] uint16, mu [A*R][L][H][D] float32, xi [A*R][L][n][H][D]
    float32, delta [A*R] int32.  Returns [A*R][L][n][H][D] uint16.
    """
    reuse = _u16(reuse)
    R, L, n, H, D = reuse.shape
    A = int(agents)
    mu = np.ascontiguousarray(mu, dtype=np.float32)
    xi = np.ascontiguousarray(xi, dtype=np.float32)
    assert mu.shape == (A * R, L, H, D) and xi.shape == (A * R, L, n, H, D)
    d = np.ascontiguousarray(delta, dtype=np.int32).reshape(A * R)
    out = np.empty((A * R, L, n, H, D), np.uint16)
    _load().oracle_compose_fresh(_p(reuse), _p(mu), _p(xi), _p(d), A, R, L, n, H, D,
                                 float(base), int(bool(rotate_keys)), _p(out))
    return out


# ------------------------------------------------------- scores and top-b

def scores(reuse, fresh, delta, agents: int, base: float, rotate_keys: bool) -> np.ndarray:
    """Check-layer divergence. reuse [R][n][H][D], fresh [A*R][n][H][D] -> [A*R][n] double."""
    reuse = _u16(reuse)
    fresh = _u16(fresh)
    R, n, H, D = reuse.shape
    A = int(agents)
    assert fresh.shape == (A * R, n, H, D)
    d = np.ascontiguousarray(delta, dtype=np.int32).reshape(A * R)
    out = np.empty((A * R, n), np.float64)
    _load().oracle_scores(_p(reuse), _p(fresh), A, R, n, H, D, _p(d), float(base),
                          int(bool(rotate_keys)), _p(out))
    return out


def topk(keys, k: int, keys_as_float: bool) -> np.ndarray:
    """Indices of the k largest keys (ties -> lower index), ascending. keys: [n]."""
    keys = np.ascontiguousarray(keys, dtype=np.float64)
    n = keys.shape[0]
    out = np.empty(max(k, 0), np.int32)
    _load().oracle_topk(_p(keys), n, int(k), int(bool(keys_as_float)), _p(out))
    return out


def ceil_ratio(num: int, den: int, n: int) -> int:
    """b = ceil(r * n) for r = num/den, in integers."""
    return -((-num * n) // den)


# --------------------------------------------------------- mean correction

def mean_correct(reuse, fresh, delta, agents: int, base: float, rotate_keys: bool, idx, w):
    """reuse [R][L][n][H][D], fresh [A*R][L][n][H][D], idx [A*R][b], w [A*R][n] ->
    (out [A*R][L][n][H][D] uint16, mu [A*R][L][H][D] double)."""
    reuse = _u16(reuse)
    fresh = _u16(fresh)
    R, L, n, H, D = reuse.shape
    A = int(agents)
    assert fresh.shape == (A * R, L, n, H, D)
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(A * R, -1)
    b = idx.shape[1]
    w = np.ascontiguousarray(w, dtype=np.float64).reshape(A * R, n)
    d = np.ascontiguousarray(delta, dtype=np.int32).reshape(A * R)
    out = np.empty_like(fresh)
    mu = np.empty((A * R, L, H, D), np.float64)
    _load().oracle_mean_correct(_p(reuse), _p(fresh), A, R, L, n, H, D, _p(d), float(base),
                                int(bool(rotate_keys)), _p(idx), b, _p(w), _p(out), _p(mu))
    return out, mu


def correct_with_weights(probe_residuals, reused, weight):
    pr = np.ascontiguousarray(probe_residuals, dtype=np.float64)
    ru = np.ascontiguousarray(reused, dtype=np.float64)
    wt = np.ascontiguousarray(weight, dtype=np.float64)
    out = np.empty_like(ru)
    mu = _load().oracle_correct_with_weights(_p(pr), pr.size, _p(ru), _p(wt), ru.size, _p(out))
    return mu, out


# ------------------------------------------------------------ low rank

def lowrank_apply(x, A, B):
    """x [C][L][n][H][D]; A [C][L][H][n][r]; B [C][L][H][r][D] (all uint16)."""
    x, A, B = _u16(x), _u16(A), _u16(B)
    C, L, n, H, D = x.shape
    r = A.shape[-1]
    assert A.shape == (C, L, H, n, r) and B.shape == (C, L, H, r, D)
    out = np.empty_like(x)
    _load().oracle_lowrank_apply(_p(x), _p(A), _p(B), C, L, n, H, D, r, _p(out))
    return out


# ------------------------------------------------------------ draft rank

def draft_scores(k, q, layer_begin: int) -> np.ndarray:
    """k [C][L][n][Hkv][D]; q [C][L][T][Hq][D] -> scores [C][n] double."""
    k, q = _u16(k), _u16(q)
    C, L, n, Hkv, D = k.shape
    _, _, T, Hq, _ = q.shape
    assert q.shape[:2] == (C, L) and q.shape[-1] == D and Hq % Hkv == 0
    out = np.empty((C, n), np.float64)
    _load().oracle_draft_scores(_p(k), _p(q), C, L, n, Hkv, D, T, Hq, int(layer_begin), _p(out))
    return out


def row_overwrite(kv, fresh, idx):
    """Return a copy of kv [C][L][n][H][D] with rows idx[c] replaced from fresh."""
    kv = _u16(kv).copy()
    fresh = _u16(fresh)
    C, L, n, H, D = kv.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(C, -1)
    _load().oracle_row_overwrite(_p(kv), _p(fresh), C, L, n, H, D, _p(idx), idx.shape[1])
    return kv


# ------------------------------------------------------- diff encode / gather

def diff_encode(master_k, master_v, sib_k, sib_v, block_tokens: int, capacity_entries=None):
    """master [L][n][H][D]; siblings [S][L][n][H][D] ->
    (mask uint32 [ceil(S*L*nblk/32)], offsets int64 [S*L*nblk+1], payload uint16
    [entries][2][bt][H][D], entries)."""
    mk, mv, sk, sv = _u16(master_k), _u16(master_v), _u16(sib_k), _u16(sib_v)
    S, L, n, H, D = sk.shape
    bt = int(block_tokens)
    nblk = n // bt
    E = S * L * nblk
    mask = np.empty((E + 31) // 32, np.uint32)
    offsets = np.empty(E + 1, np.int64)
    if capacity_entries is None:
        capacity_entries = E
    payload = np.empty((max(int(capacity_entries), 1), 2, bt, H, D), np.uint16)
    total = _load().oracle_diff_encode(_p(mk), _p(mv), _p(sk), _p(sv), S, L, n, H, D, bt,
                                       _p(mask), _p(offsets), _p(payload), int(capacity_entries))
    return mask, offsets, payload[:total], int(total)


def diff_gather(master_k, master_v, mask, offsets, payload, siblings: int, block_tokens: int):
    mk, mv = _u16(master_k), _u16(master_v)
    L, n, H, D = mk.shape
    S = int(siblings)
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    payload = _u16(payload) if payload.size else np.zeros((1,), np.uint16)
    ok = np.empty((S, L, n, H, D), np.uint16)
    ov = np.empty_like(ok)
    _load().oracle_diff_gather(_p(mk), _p(mv), _p(mask), _p(offsets), _p(payload), S, L, n, H, D,
                               int(block_tokens), _p(ok), _p(ov))
    return ok, ov


def diff_restore(master_k, master_v, mask, offsets, payload, siblings: int, block_tokens: int, delta,
                 rope_base: float, slot_map, pool_k, pool_v):
    """Restore every mirror into the paged pool (pool_k/pool_v [L][slots][H][D], updated in
    place and returned): token t of mirror s goes to slot slot_map[s][t] (< 0: skipped),
    keys rotated by delta[s]."""
    mk, mv = _u16(master_k), _u16(master_v)
    L, n, H, D = mk.shape
    S = int(siblings)
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    payload = _u16(payload) if payload.size else np.zeros((1,), np.uint16)
    delta = np.ascontiguousarray(delta, dtype=np.int32)
    slot_map = np.ascontiguousarray(slot_map, dtype=np.int32).reshape(S, n)
    pk = np.array(pool_k, dtype=np.uint16, order="C", copy=True)
    pv = np.array(pool_v, dtype=np.uint16, order="C", copy=True)
    assert pk.shape[0] == L and pk.shape[2:] == (H, D) and pv.shape == pk.shape
    _load().oracle_diff_restore(_p(mk), _p(mv), _p(mask), _p(offsets), _p(payload), S, L, n, H, D,
                                int(block_tokens), _p(delta), float(rope_base), _p(slot_map),
                                int(pk.shape[1]), _p(pk), _p(pv))
    return pk, pv


# ------------------------------------------------------------ anchor-pool correction

def anchor_gate(v_src, a_c, b_ct, k: int, T: float = 1.0, tau: float = 0.5):
    """v_src [C][L][n][F] uint16; a_c [C][V][L][n][r]; b_ct [C][V][L][F][r] ->
    (d [C][V], g [C][V], hbar [C], accept [C] bool)."""
    x, a, b = _u16(v_src), _u16(a_c), _u16(b_ct)
    C, L, n, F = x.shape
    V, r = a.shape[1], a.shape[-1]
    assert a.shape == (C, V, L, n, r) and b.shape == (C, V, L, F, r)
    d = np.empty((C, V), np.float64)
    g = np.empty_like(d)
    hbar = np.empty(C, np.float64)
    acc = np.empty(C, np.int32)
    _load().oracle_anchor_gate(_p(x), _p(a), _p(b), C, V, L, n, F, r, int(k), float(T), float(tau),
                               _p(d), _p(g), _p(hbar), _p(acc))
    return d, g, hbar, acc.astype(bool)


def anchor_weights(x, a_c, b_ct, T: float = 1.0):
    """x [C][L][n][F] uint16 (one plane); a_c [C][V][L][n][r]; b_ct [C][V][L][F][r] ->
    w [C][L][n][V] float64."""
    x, a, b = _u16(x), _u16(a_c), _u16(b_ct)
    C, L, n, F = x.shape
    V, r = a.shape[1], a.shape[-1]
    assert a.shape == (C, V, L, n, r) and b.shape == (C, V, L, F, r)
    w = np.empty((C, L, n, V), np.float64)
    _load().oracle_anchor_weights(_p(x), _p(a), _p(b), C, V, L, n, F, r, float(T), _p(w))
    return w


def anchor_correct(x, a_d, b_dt, w, heads: int, delta, rope_base: float, rotate: bool):
    """x [C][L][n][H*D] uint16; a_d [C][V][L][n][r]; b_dt [C][V][L][H*D][r]; w [C][L][n][V]
    -> out uint16 like x."""
    x, a, b = _u16(x), _u16(a_d), _u16(b_dt)
    C, L, n, F = x.shape
    V, r = a.shape[1], a.shape[-1]
    H = int(heads)
    assert F % H == 0 and a.shape == (C, V, L, n, r) and b.shape == (C, V, L, F, r)
    w = np.ascontiguousarray(w, dtype=np.float64).reshape(C, L, n, V)
    dl = np.ascontiguousarray(delta, dtype=np.int32).reshape(C)
    out = np.empty_like(x)
    _load().oracle_anchor_correct(_p(x), _p(a), _p(b), _p(w), C, V, L, n, H, F // H, r, _p(dl),
                                  float(rope_base), int(bool(rotate)), _p(out))
    return out


# ------------------------------------------------------------ repair layouts

LAYOUT_SINGLE, LAYOUT_CHUNK, LAYOUT_GROW = 0, 1, 2


def repair_layout(scores, layout: int, chunk_tokens: int = 64, budget=(1, 5), tau: float = 0.25,
                  skip: bool = True, max_rows=None):
    """scores [U][n] float64 -> (idx [U][max_rows] int32 ascending then -1, counts [U])."""
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    if sc.ndim == 1:
        sc = sc[None]
    U, n = sc.shape
    max_rows = n if max_rows is None else int(max_rows)
    idx = np.empty((U, max(max_rows, 1)), np.int32)
    counts = np.empty(U, np.int32)
    _load().oracle_repair_layout(_p(sc), U, n, int(layout), int(chunk_tokens), int(budget[0]), int(budget[1]),
                                 float(tau), int(bool(skip)), _p(idx), max(max_rows, 1), _p(counts))
    return idx[:, :max_rows], counts


# ------------------------------------------------------------ master selection, split diffs

def master_select(d_k, d_v, agents: int):
    """d_k, d_v [A*R][n] float32 (either may be None) -> (master, totals [A] float64)."""
    ref = d_k if d_k is not None else d_v
    ref = np.ascontiguousarray(ref, dtype=np.float32)
    A = int(agents)
    R = ref.shape[0] // A
    n = ref.shape[-1]
    dk = None if d_k is None else np.ascontiguousarray(d_k, dtype=np.float32)
    dv = None if d_v is None else np.ascontiguousarray(d_v, dtype=np.float32)
    tot = np.empty(A, np.float64)
    m = _load().oracle_master_select(None if dk is None else _p(dk), None if dv is None else _p(dv), A, R, n,
                                     _p(tot))
    return int(m), tot


def diff_encode_split(master_k, master_v, sib_k, sib_v, block_tokens: int):
    """-> per plane (mask uint32, offsets int64 [E+1], payload [entries][bt][H][D]) for K and V."""
    mk, mv, sk, sv = _u16(master_k), _u16(master_v), _u16(sib_k), _u16(sib_v)
    S, L, n, H, D = sk.shape
    bt = int(block_tokens)
    E = S * L * (n // bt)
    masks = [np.empty((E + 31) // 32, np.uint32) for _ in range(2)]
    offs = [np.empty(E + 1, np.int64) for _ in range(2)]
    pays = [np.empty((E, bt, H, D), np.uint16) for _ in range(2)]
    cap = np.array([E, E], np.int64)
    need = np.zeros(2, np.int64)
    _load().oracle_diff_encode_split(_p(mk), _p(mv), _p(sk), _p(sv), S, L, n, H, D, bt, _p(masks[0]), _p(masks[1]),
                                     _p(offs[0]), _p(offs[1]), _p(pays[0]), _p(pays[1]), _p(cap), _p(need))
    return ((masks[0], offs[0], pays[0][:need[0]]), (masks[1], offs[1], pays[1][:need[1]]))


def diff_gather_split(master_k, master_v, k_diff, v_diff, siblings: int, block_tokens: int):
    mk, mv = _u16(master_k), _u16(master_v)
    L, n, H, D = mk.shape
    S = int(siblings)
    parts = []
    for mask, off, pay in (k_diff, v_diff):
        pay = _u16(pay) if pay.size else np.zeros((1,), np.uint16)
        parts.append((np.ascontiguousarray(mask, dtype=np.uint32), np.ascontiguousarray(off, dtype=np.int64), pay))
    ok = np.empty((S, L, n, H, D), np.uint16)
    ov = np.empty_like(ok)
    (mk_, ok_, pk_), (mv_, ov_, pv_) = parts
    _load().oracle_diff_gather_split(_p(mk), _p(mv), _p(mk_), _p(mv_), _p(ok_), _p(ov_), _p(pk_), _p(pv_), S, L, n,
                                     H, D, int(block_tokens), _p(ok), _p(ov))
    return ok, ov
