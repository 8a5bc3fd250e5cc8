"""ctypes binding of libkvfix (include/kvfix.h).

Argument marshalling only: every function checks tensor dtypes/devices, builds the
plane descriptors from tensor shapes and strides, allocates outputs with torch on the
tensors' device and calls the C entry point of the same name on the current CUDA
stream.  All arithmetic runs in the library's CUDA kernels.  If libkvfix.so is
missing, importing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvfix.so")

OK, EINVAL, ENOSPACE, ECUDA, ETIMEOUT, EDEVICE = range(6)
STATUS_NAMES = {0: "KVFIX_OK", 1: "KVFIX_EINVAL", 2: "KVFIX_ENOSPACE", 3: "KVFIX_ECUDA",
                4: "KVFIX_ETIMEOUT", 5: "KVFIX_EDEVICE"}


class KvfixError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class KvDesc(ctypes.Structure):
    _fields_ = [("chunks", ctypes.c_int32), ("layers", ctypes.c_int32), ("tokens", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("stride_chunk", ctypes.c_int64), ("stride_layer", ctypes.c_int64),
                ("stride_token", ctypes.c_int64)]


# name -> (restype, argtypes); mirrors include/kvfix.h
P, I32, I64, F64, SZ, D = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double,
                           ctypes.c_size_t, KvDesc)
SIGNATURES = {
    "kvfix_version": (ctypes.c_int, []),
    "kvfix_last_error": (ctypes.c_char_p, []),
    "kvfix_check_status": (ctypes.c_int, [P]),
    "kvfix_rerope": (ctypes.c_int, [P, D, P, D, P, F64, P]),
    "kvfix_score_topk": (ctypes.c_int, [P, P, D, P, P, D, I32, P, F64, I32, P, P, P, P, P, P, P, P, P, P]),
    "kvfix_mean_correct": (ctypes.c_int, [P, P, D, P, P, D, P, P, D, I32, P, F64, P, P, I32, P, P, P, P, P]),
    "kvfix_lowrank_apply": (ctypes.c_int, [P, D, P, P, I32, P, D, P]),
    "kvfix_draft_rank_workspace_bytes": (SZ, [D, I32]),
    "kvfix_draft_rank": (ctypes.c_int, [P, D, P, I32, I32, I32, I32, P, P, P, P, D, P, P, P, SZ, P]),
    "kvfix_draft_rank_noalloc": (ctypes.c_int, [P, D, P, I32, I32, I32, I32, P, P, P, P, D, P, P, P]),
    "kvfix_lowrank_draft_workspace_bytes": (SZ, [D, I32]),
    "kvfix_lowrank_draft": (ctypes.c_int, [P, D, P, P, I32, P, D, P, I32, I32, I32, I32, P, P, P, P, D, P, P, SZ, P]),
    "kvfix_diff_encode": (ctypes.c_int, [P, P, D, P, P, D, I32, P, P, P, I64, P, P]),
    "kvfix_diff_gather": (ctypes.c_int, [P, P, D, P, P, P, I64, I32, I32, P, P, D, P]),
    "kvfix_diff_restore": (ctypes.c_int, [P, P, D, P, P, P, I64, I32, I32, P, F64, P, P, P, D, P]),
    "kvfix_repair_layout": (ctypes.c_int, [P, I32, I32, I32, I32, I32, I32, F64, I32, P, I32, P, P]),
    "kvfix_master_select": (ctypes.c_int, [P, P, I32, I32, I32, P, P, P]),
    "kvfix_selftest_wait": (ctypes.c_int, [I64, P, P]),
    "kvfix_anchor_gate_correct": (ctypes.c_int, [P, P, D, P, P, P, P, P, P, P, P, I32, I32, I32, F64, F64, P, F64, P,
                                                 P, P, P, P, P, P, P, D, P, SZ, P]),
    "kvfix_diff_encode_split": (ctypes.c_int, [P, P, D, P, P, D, I32, P, P, P, P, P, P, I64, I64, P, P]),
    "kvfix_diff_gather_split": (ctypes.c_int, [P, P, D, P, P, P, P, P, P, I64, I64, I32, I32, P, P, D, P]),
    "kvfix_diff_restore_split": (ctypes.c_int, [P, P, D, P, P, P, P, P, P, I64, I64, I32, I32, P, F64, P, P, P, D,
                                                P]),
    "kvfix_repair_rows": (ctypes.c_int, [P, P, D, P, P, D, P, I32, P, P]),
    "kvfix_anchor_gate_workspace_bytes": (SZ, [D, I32, I32]),
    "kvfix_anchor_gate": (ctypes.c_int, [P, D, P, P, I32, I32, I32, F64, F64, P, P, P, P, P, SZ, P]),
    "kvfix_anchor_correct": (ctypes.c_int, [P, P, D, P, P, P, P, P, P, P, P, I32, I32, F64, P, F64, P, P, P, P, P,
                                            D, P]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _check(status: int):
    if status != OK:
        raise KvfixError(status, lib.kvfix_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _bf16(t, name):
    if t is None:
        return
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor (got {t.dtype} on {t.device})")


def plane_desc(t: torch.Tensor) -> KvDesc:
    """Descriptor of a [chunks][layers][tokens][heads][dim] (or [chunks][tokens][heads][dim],
    read as one layer) bf16 view whose heads and dims are contiguous."""
    if t.dim() == 4:
        t = t.unsqueeze(1)
    if t.dim() != 5:
        raise ValueError(f"KV plane must be 4-D or 5-D, got shape {tuple(t.shape)}")
    C, L, n, H, Dh = t.shape
    sc, sl, st, sh, sd = t.stride()
    if (sd != 1 or sh != Dh) and H * Dh > 1:
        raise ValueError("KV plane views need contiguous heads and dims (stride(-1) == 1, "
                         "stride(-2) == head_dim)")
    return KvDesc(C, L, n, H, Dh, sc if C > 1 else 0, sl if L > 1 else 0, st if n > 1 else H * Dh)


def _i32(t, name):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA int32 tensor")


def _f32(t, name):
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA float32 tensor")


def version() -> int:
    return lib.kvfix_version()


def check_status(stream_of: torch.Tensor | None = None) -> int:
    """Synchronise the current stream and raise if the device flagged a condition."""
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _check(lib.kvfix_check_status(s))
    return OK


# --------------------------------------------------------------------- calls

def rerope(k: torch.Tensor, delta: torch.Tensor, rope_base: float, out: torch.Tensor | None = None):
    _bf16(k, "k")
    _i32(delta, "delta")
    out = torch.empty_like(k) if out is None else out
    _bf16(out, "out")
    _check(lib.kvfix_rerope(_ptr(k), plane_desc(k), _ptr(out), plane_desc(out), _ptr(delta),
                            float(rope_base), _stream(k)))
    return out


def score_topk(k_reuse, v_reuse, k_fresh, v_fresh, agents: int, delta, rope_base: float, b: int,
               masks: bool = False):
    """Check-layer views: reuse [R](1)[n][H][D], fresh [agents*R](1)[n][H][D]."""
    for t, nm in ((k_reuse, "k_reuse"), (v_reuse, "v_reuse"), (k_fresh, "k_fresh"), (v_fresh, "v_fresh")):
        _bf16(t, nm)
    _i32(delta, "delta")
    rd, fd = plane_desc(k_reuse), plane_desc(k_fresh)
    units, n = fd.chunks, fd.tokens
    dev = k_reuse.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"d_k": torch.empty(units, n, **f32), "d_v": torch.empty(units, n, **f32),
           "w_k": torch.empty(units, n, **f32), "w_v": torch.empty(units, n, **f32),
           "idx_k": torch.empty(units, max(b, 0), dtype=torch.int32, device=dev),
           "idx_v": torch.empty(units, max(b, 0), dtype=torch.int32, device=dev)}
    words = (n + 31) // 32
    if masks:
        for nm in ("mask_k", "mask_v", "mask_union"):
            out[nm] = torch.empty(units, words, dtype=torch.int32, device=dev)
    _check(lib.kvfix_score_topk(_ptr(k_reuse), _ptr(v_reuse), rd, _ptr(k_fresh), _ptr(v_fresh), fd,
                                int(agents), _ptr(delta), float(rope_base), int(b),
                                _ptr(out["d_k"]), _ptr(out["d_v"]), _ptr(out["w_k"]), _ptr(out["w_v"]),
                                _ptr(out["idx_k"]) if b > 0 else None, _ptr(out["idx_v"]) if b > 0 else None,
                                _ptr(out.get("mask_k")), _ptr(out.get("mask_v")),
                                _ptr(out.get("mask_union")), _stream(k_reuse)))
    return out


def mean_correct(k_reuse, v_reuse, k_fresh, v_fresh, agents: int, delta, rope_base: float,
                 idx_k, idx_v, w_k, w_v, k_out=None, v_out=None, mu_k=None, mu_v=None):
    """reuse [R][L][n][H][D]; fresh/out [agents*R][L][n][H][D]; idx [agents*R][b]."""
    for t, nm in ((k_reuse, "k_reuse"), (v_reuse, "v_reuse"), (k_fresh, "k_fresh"), (v_fresh, "v_fresh")):
        _bf16(t, nm)
    _i32(delta, "delta")
    _i32(idx_k, "idx_k")
    _i32(idx_v, "idx_v")
    _f32(w_k, "w_k")
    _f32(w_v, "w_v")
    if idx_k.shape != idx_v.shape:
        raise ValueError("idx_k and idx_v must have the same shape")
    b = idx_k.shape[-1] if idx_k.dim() else 0
    k_out = torch.empty_like(k_fresh) if k_out is None else k_out
    v_out = torch.empty_like(v_fresh) if v_out is None else v_out
    rd, fd, od = plane_desc(k_reuse), plane_desc(k_fresh), plane_desc(k_out)
    units, L, H, Dh = fd.chunks, fd.layers, fd.kv_heads, fd.head_dim
    if mu_k is None:
        mu_k = torch.empty(units, L, H * Dh, dtype=torch.float32, device=k_reuse.device)
    if mu_v is None:
        mu_v = torch.empty(units, L, H * Dh, dtype=torch.float32, device=k_reuse.device)
    _check(lib.kvfix_mean_correct(_ptr(k_reuse), _ptr(v_reuse), rd, _ptr(k_fresh), _ptr(v_fresh), fd,
                                  _ptr(k_out), _ptr(v_out), od, int(agents), _ptr(delta),
                                  float(rope_base), _ptr(idx_k), _ptr(idx_v), int(b), _ptr(w_k),
                                  _ptr(w_v), _ptr(mu_k), _ptr(mu_v), _stream(k_reuse)))
    return k_out, v_out, mu_k, mu_v


def lowrank_apply(x, A, B, out=None):
    """x [C][L][n][H][D]; A [C][L][H][n][r]; B [C][L][H][r][D] (A, B contiguous)."""
    _bf16(x, "x")
    _bf16(A, "A")
    _bf16(B, "B")
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous")
    out = torch.empty_like(x) if out is None else out
    _bf16(out, "out")
    _check(lib.kvfix_lowrank_apply(_ptr(x), plane_desc(x), _ptr(A), _ptr(B), int(A.shape[-1]), _ptr(out),
                                   plane_desc(out), _stream(x)))
    return out


def draft_rank_workspace_bytes(k, layer_begin: int) -> int:
    return int(lib.kvfix_draft_rank_workspace_bytes(plane_desc(k), int(layer_begin)))


def draft_rank(k, q, layer_begin: int, k_rows: int, k_fresh=None, v_fresh=None, k_io=None,
               v_io=None, workspace=None):
    """k [C][L][n][Hkv][D]; q [C][L][T][Hq][D] contiguous.  Returns (idx, scores)."""
    _bf16(k, "k")
    _bf16(q, "q")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    d = plane_desc(k)
    C, n = d.chunks, d.tokens
    ws_bytes = draft_rank_workspace_bytes(k, layer_begin)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=k.device)
    idx = torch.empty(C, max(k_rows, 0), dtype=torch.int32, device=k.device)
    scores = torch.empty(C, n, dtype=torch.float64, device=k.device)
    fd = plane_desc(k_fresh) if k_fresh is not None else (plane_desc(v_fresh) if v_fresh is not None else d)
    _check(lib.kvfix_draft_rank(_ptr(k), d, _ptr(q), int(q.shape[2]), int(q.shape[3]), int(layer_begin),
                                int(k_rows), _ptr(idx), _ptr(scores), _ptr(k_fresh), _ptr(v_fresh), fd,
                                _ptr(k_io), _ptr(v_io), _ptr(workspace), workspace.numel(), _stream(k)))
    return idx, scores


def lowrank_draft_workspace_bytes(k, layer_begin: int) -> int:
    return int(lib.kvfix_lowrank_draft_workspace_bytes(plane_desc(k), int(layer_begin)))


def lowrank_draft(x, A, B, q, layer_begin: int, k_rows: int, out=None, k_fresh=None, v_fresh=None, v_io=None,
                  workspace=None):
    """out = x + A B (the key plane) and the draft ranking of out in one pass; with k_fresh
    the selected rows of out, with v_fresh/v_io those of v_io, are overwritten.  x, out
    [C][L][n][Hkv][D]; A [C][L][Hkv][n][r]; B [C][L][Hkv][r][D]; q [C][L][T][Hq][D].
    Returns (out, idx, scores)."""
    for t, nm in ((x, "x"), (A, "A"), (B, "B"), (q, "q")):
        _bf16(t, nm)
    if not (A.is_contiguous() and B.is_contiguous() and q.is_contiguous()):
        raise ValueError("A, B and q must be contiguous")
    out = torch.empty_like(x) if out is None else out
    _bf16(out, "out")
    d, od = plane_desc(x), plane_desc(out)
    C, n = d.chunks, d.tokens
    ws_bytes = lowrank_draft_workspace_bytes(out, layer_begin)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    idx = torch.empty(C, max(k_rows, 0), dtype=torch.int32, device=x.device)
    scores = torch.empty(C, n, dtype=torch.float64, device=x.device)
    fd = plane_desc(k_fresh) if k_fresh is not None else (plane_desc(v_fresh) if v_fresh is not None else d)
    _check(lib.kvfix_lowrank_draft(_ptr(x), d, _ptr(A), _ptr(B), int(A.shape[-1]), _ptr(out), od, _ptr(q),
                                   int(q.shape[2]), int(q.shape[3]), int(layer_begin), int(k_rows), _ptr(idx),
                                   _ptr(scores), _ptr(k_fresh), _ptr(v_fresh), fd, _ptr(v_io), _ptr(workspace),
                                   workspace.numel(), _stream(x)))
    return out, idx, scores


def diff_encode(master_k, master_v, sib_k, sib_v, block_tokens: int, capacity: int | None = None,
                sync: bool = True):
    """master [L][n][H][D] (or [1][L][n][H][D]); siblings [S][L][n][H][D].
    Returns (mask int32 words, offsets int64, payload [cap][2][bt][H][D], entries or None)."""
    for t, nm in ((master_k, "master_k"), (master_v, "master_v"), (sib_k, "sib_k"), (sib_v, "sib_v")):
        _bf16(t, nm)
    mk = master_k.unsqueeze(0) if master_k.dim() == 4 else master_k
    mv = master_v.unsqueeze(0) if master_v.dim() == 4 else master_v
    md, sd = plane_desc(mk), plane_desc(sib_k)
    S, L, n, H, Dh = sd.chunks, sd.layers, sd.tokens, sd.kv_heads, sd.head_dim
    bt = int(block_tokens)
    E = S * L * (n // bt)
    dev = sib_k.device
    mask = torch.empty((E + 31) // 32, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int64, device=dev)
    cap = E if capacity is None else int(capacity)
    payload = torch.empty(max(cap, 1), 2, bt, H, Dh, dtype=torch.bfloat16, device=dev)
    entries = ctypes.c_int64(-1)
    st = lib.kvfix_diff_encode(_ptr(mk), _ptr(mv), md, _ptr(sib_k), _ptr(sib_v), sd, bt, _ptr(mask),
                               _ptr(offsets), _ptr(payload), cap, ctypes.byref(entries) if sync else None,
                               _stream(sib_k))
    _check(st)
    return mask, offsets, payload, (entries.value if sync else None)


def diff_gather(master_k, master_v, mask, offsets, payload, siblings: int, block_tokens: int,
                out_k=None, out_v=None, payload_entries: int | None = None):
    _bf16(master_k, "master_k")
    _bf16(master_v, "master_v")
    mk = master_k.unsqueeze(0) if master_k.dim() == 4 else master_k
    mv = master_v.unsqueeze(0) if master_v.dim() == 4 else master_v
    md = plane_desc(mk)
    shape = (int(siblings),) + tuple(mk.shape[1:])
    out_k = torch.empty(shape, dtype=torch.bfloat16, device=mk.device) if out_k is None else out_k
    out_v = torch.empty(shape, dtype=torch.bfloat16, device=mk.device) if out_v is None else out_v
    pe = payload.shape[0] if payload_entries is None else int(payload_entries)
    _check(lib.kvfix_diff_gather(_ptr(mk), _ptr(mv), md, _ptr(mask), _ptr(offsets), _ptr(payload), pe,
                                 int(siblings), int(block_tokens), _ptr(out_k), _ptr(out_v),
                                 plane_desc(out_k), _stream(mk)))
    return out_k, out_v


def diff_restore(master_k, master_v, mask, offsets, payload, siblings: int, block_tokens: int,
                 delta, rope_base: float, slot_mapping, pool_k, pool_v,
                 payload_entries: int | None = None):
    """Restore every sibling into the paged pool pool_k/pool_v [layers][slots][heads][dim]
    (written in place): token t of sibling s goes to row slot_mapping[s][t] (< 0: not
    restored), keys rotated by delta[s]."""
    _bf16(master_k, "master_k")
    _bf16(master_v, "master_v")
    _bf16(pool_k, "pool_k")
    _bf16(pool_v, "pool_v")
    _i32(delta, "delta")
    _i32(slot_mapping, "slot_mapping")
    mk = master_k.unsqueeze(0) if master_k.dim() == 4 else master_k
    mv = master_v.unsqueeze(0) if master_v.dim() == 4 else master_v
    if pool_k.dim() != 4 or pool_v.shape != pool_k.shape:
        raise ValueError("pool_k and pool_v must both be [layers][slots][heads][dim]")
    if delta.numel() != int(siblings) or slot_mapping.numel() != int(siblings) * mk.shape[2]:
        raise ValueError("delta must hold one shift per sibling and slot_mapping one slot per "
                         "(sibling, token)")
    pe = payload.shape[0] if payload_entries is None else int(payload_entries)
    _check(lib.kvfix_diff_restore(_ptr(mk), _ptr(mv), plane_desc(mk), _ptr(mask), _ptr(offsets),
                                  _ptr(payload), pe, int(siblings), int(block_tokens), _ptr(delta),
                                  float(rope_base), _ptr(slot_mapping), _ptr(pool_k), _ptr(pool_v),
                                  plane_desc(pool_k.unsqueeze(0)), _stream(mk)))
    return pool_k, pool_v


def _factor(t, name, shape):
    _bf16(t, name)
    if not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous tensor of shape {tuple(shape)}, got {tuple(t.shape)}")


def anchor_gate(v_src, a_c, b_ct, prefix: int, temperature: float = 1.0, tau: float = 0.5):
    """Reliability gate per segment.  v_src [C][L][n][H][D]; a_c [C][V][L][n][r];
    b_ct [C][V][L][H*D][r].  Returns (d [C][V] f64, g [C][V] f64, hbar [C] f64, accept [C] i32)."""
    _bf16(v_src, "v_src")
    x = v_src if v_src.dim() == 5 else v_src.unsqueeze(0)
    C, L, n, H, Dh = x.shape
    V, r = a_c.shape[1], a_c.shape[-1]
    _factor(a_c, "a_c", (C, V, L, n, r))
    _factor(b_ct, "b_ct", (C, V, L, H * Dh, r))
    dev = x.device
    d = torch.empty((C, V), dtype=torch.float64, device=dev)
    g = torch.empty_like(d)
    hbar = torch.empty(C, dtype=torch.float64, device=dev)
    acc = torch.empty(C, dtype=torch.int32, device=dev)
    desc = plane_desc(x)
    nbytes = lib.kvfix_anchor_gate_workspace_bytes(desc, V, int(prefix))
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _check(lib.kvfix_anchor_gate(_ptr(x), desc, _ptr(a_c), _ptr(b_ct), V, r, int(prefix), float(temperature),
                                 float(tau), _ptr(d), _ptr(g), _ptr(hbar), _ptr(acc), _ptr(ws), ws.numel(),
                                 _stream(x)))
    return d, g, hbar, acc


def anchor_correct(k_src, v_src, factors: dict, delta, rope_base: float, temperature: float = 1.0,
                   accept=None, out_k=None, out_v=None, w_k=None, w_v=None):
    """Token-weighted anchor correction of both planes.  k_src/v_src [C][L][n][H][D];
    factors: a_c_k, b_ct_k, a_c_v, b_ct_v, a_d_k, b_dt_k, a_d_v, b_dt_v ([C][V][L][n][r] and
    [C][V][L][H*D][r]).  Returns (out_k, out_v, w_k, w_v); w_* [C][L][n][V] float32."""
    _bf16(k_src, "k_src")
    _bf16(v_src, "v_src")
    _i32(delta, "delta")
    C, L, n, H, Dh = k_src.shape
    V, r = factors["a_c_k"].shape[1], factors["a_c_k"].shape[-1]
    names = ("a_c_k", "b_ct_k", "a_c_v", "b_ct_v", "a_d_k", "b_dt_k", "a_d_v", "b_dt_v")
    for nm in names:
        _factor(factors[nm], nm, (C, V, L, n, r) if nm.startswith("a_") else (C, V, L, H * Dh, r))
    dev = k_src.device
    out_k = torch.empty_like(k_src) if out_k is None else out_k
    out_v = torch.empty_like(v_src) if out_v is None else out_v
    w_k = torch.empty((C, L, n, V), dtype=torch.float32, device=dev) if w_k is None else w_k
    w_v = torch.empty((C, L, n, V), dtype=torch.float32, device=dev) if w_v is None else w_v
    _f32(w_k, "w_k")
    _f32(w_v, "w_v")
    if accept is not None:
        _i32(accept, "accept")
    _check(lib.kvfix_anchor_correct(_ptr(k_src), _ptr(v_src), plane_desc(k_src),
                                    *[_ptr(factors[nm]) for nm in names], V, r, float(temperature), _ptr(delta),
                                    float(rope_base), _ptr(accept), _ptr(w_k), _ptr(w_v), _ptr(out_k), _ptr(out_v),
                                    plane_desc(out_k), _stream(k_src)))
    return out_k, out_v, w_k, w_v


LAYOUT_SINGLE, LAYOUT_CHUNK, LAYOUT_GROW = 0, 1, 2


def _round_half_even(p: int, q: int) -> int:
    f, r = divmod(p, q)
    return f + (1 if 2 * r > q or (2 * r == q and f % 2) else 0)


def layout_max_rows(tokens: int, layout: int, chunk_tokens: int = 64, budget=(1, 5)) -> int:
    """The most rows a layout can choose (the size idx needs per unit)."""
    num, den = budget
    if layout == LAYOUT_CHUNK:
        nch = -(-tokens // chunk_tokens)
        c = min(nch, max(1, _round_half_even(num * tokens, den * chunk_tokens)))
        return max(1, min(tokens, c * chunk_tokens))
    return max(1, _round_half_even(num * tokens, den))


def repair_layout(scores, layout: int, chunk_tokens: int = 64, budget=(1, 5), tau: float = 0.25,
                  skip_rule: bool = True, max_rows: int | None = None):
    """scores [units][tokens] float64 (CUDA) -> (idx [units][max_rows] int32, counts [units] int32)."""
    if scores.dtype != torch.float64 or not scores.is_cuda or not scores.is_contiguous():
        raise TypeError("scores must be a contiguous CUDA float64 tensor")
    sc = scores if scores.dim() == 2 else scores.unsqueeze(0)
    U, n = sc.shape
    mr = layout_max_rows(n, layout, chunk_tokens, budget) if max_rows is None else int(max_rows)
    idx = torch.empty((U, mr), dtype=torch.int32, device=sc.device)
    counts = torch.empty(U, dtype=torch.int32, device=sc.device)
    _check(lib.kvfix_repair_layout(_ptr(sc), U, n, int(layout), int(chunk_tokens), int(budget[0]), int(budget[1]),
                                   float(tau), int(bool(skip_rule)), _ptr(idx), mr, _ptr(counts), _stream(sc)))
    return idx, counts


def repair_rows(k_io, v_io, k_fresh, v_fresh, idx, counts):
    """Overwrite rows idx[c][:counts[c]] of k_io / v_io ([C][L][n][H][D]) with the fresh rows."""
    for t, nm in ((k_io, "k_io"), (v_io, "v_io"), (k_fresh, "k_fresh"), (v_fresh, "v_fresh")):
        _bf16(t, nm)
    _i32(idx, "idx")
    _i32(counts, "counts")
    ref = k_io if k_io is not None else v_io
    fref = k_fresh if k_fresh is not None else v_fresh
    _check(lib.kvfix_repair_rows(_ptr(k_io), _ptr(v_io), plane_desc(ref), _ptr(k_fresh), _ptr(v_fresh),
                                 plane_desc(fref), _ptr(idx), idx.shape[-1], _ptr(counts), _stream(ref)))


def master_select(d_k, d_v, agents: int):
    """d_k, d_v [agents*R][n] float32 (CUDA; either may be None) -> (master int32 [1], totals [agents] f64)."""
    ref = d_k if d_k is not None else d_v
    for t, nm in ((d_k, "d_k"), (d_v, "d_v")):
        if t is not None:
            _f32(t, nm)
    A = int(agents)
    R = ref.shape[0] // A
    totals = torch.empty(A, dtype=torch.float64, device=ref.device)
    master = torch.empty(1, dtype=torch.int32, device=ref.device)
    _check(lib.kvfix_master_select(_ptr(d_k), _ptr(d_v), A, R, ref.shape[-1], _ptr(totals), _ptr(master),
                                   _stream(ref)))
    return master, totals


def diff_encode_split(master_k, master_v, sib_k, sib_v, block_tokens: int, capacity=None, sync: bool = True):
    """Per-plane block lists.  Returns ((mask_k, offsets_k, payload_k), (mask_v, offsets_v, payload_v),
    (entries_k, entries_v) or None); payload_P [cap][bt][H][D]."""
    for t, nm in ((master_k, "master_k"), (master_v, "master_v"), (sib_k, "sib_k"), (sib_v, "sib_v")):
        _bf16(t, nm)
    mk = master_k.unsqueeze(0) if master_k.dim() == 4 else master_k
    mv = master_v.unsqueeze(0) if master_v.dim() == 4 else master_v
    md, sd = plane_desc(mk), plane_desc(sib_k)
    S, L, n, H, Dh = sd.chunks, sd.layers, sd.tokens, sd.kv_heads, sd.head_dim
    bt = int(block_tokens)
    E = S * L * (n // bt)
    dev = sib_k.device
    caps = (E, E) if capacity is None else tuple(int(c) for c in capacity)
    lists = []
    for cap in caps:
        lists.append((torch.empty((E + 31) // 32, dtype=torch.int32, device=dev),
                      torch.empty(E + 1, dtype=torch.int64, device=dev),
                      torch.empty(max(cap, 1), bt, H, Dh, dtype=torch.bfloat16, device=dev)))
    entries = (ctypes.c_int64 * 2)(-1, -1)
    (mk_, ok_, pk_), (mv_, ov_, pv_) = lists
    _check(lib.kvfix_diff_encode_split(_ptr(mk), _ptr(mv), md, _ptr(sib_k), _ptr(sib_v), sd, bt, _ptr(mk_), _ptr(mv_),
                                       _ptr(ok_), _ptr(ov_), _ptr(pk_), _ptr(pv_), caps[0], caps[1],
                                       entries if sync else None, _stream(sib_k)))
    return lists[0], lists[1], ((entries[0], entries[1]) if sync else None)


def diff_gather_split(master_k, master_v, k_list, v_list, siblings: int, block_tokens: int, out_k=None,
                      out_v=None, entries=None):
    _bf16(master_k, "master_k")
    _bf16(master_v, "master_v")
    mk = master_k.unsqueeze(0) if master_k.dim() == 4 else master_k
    mv = master_v.unsqueeze(0) if master_v.dim() == 4 else master_v
    md = plane_desc(mk)
    shape = (int(siblings),) + tuple(mk.shape[1:])
    out_k = torch.empty(shape, dtype=torch.bfloat16, device=mk.device) if out_k is None else out_k
    out_v = torch.empty(shape, dtype=torch.bfloat16, device=mk.device) if out_v is None else out_v
    ek, ev = (k_list[2].shape[0], v_list[2].shape[0]) if entries is None else entries
    _check(lib.kvfix_diff_gather_split(_ptr(mk), _ptr(mv), md, _ptr(k_list[0]), _ptr(v_list[0]), _ptr(k_list[1]),
                                       _ptr(v_list[1]), _ptr(k_list[2]), _ptr(v_list[2]), int(ek), int(ev),
                                       int(siblings), int(block_tokens), _ptr(out_k), _ptr(out_v), plane_desc(out_k),
                                       _stream(mk)))
    return out_k, out_v


def diff_restore_split(master_k, master_v, k_list, v_list, siblings: int, block_tokens: int, delta,
                       rope_base: float, slot_mapping, pool_k, pool_v, entries=None):
    """diff_restore from the per-plane lists of diff_encode_split (written in place)."""
    for t, name in ((master_k, "master_k"), (master_v, "master_v"), (pool_k, "pool_k"), (pool_v, "pool_v")):
        _bf16(t, name)
    _i32(delta, "delta")
    _i32(slot_mapping, "slot_mapping")
    mk = master_k.unsqueeze(0) if master_k.dim() == 4 else master_k
    mv = master_v.unsqueeze(0) if master_v.dim() == 4 else master_v
    if pool_k.dim() != 4 or pool_v.shape != pool_k.shape:
        raise ValueError("pool_k and pool_v must both be [layers][slots][heads][dim]")
    if delta.numel() != int(siblings) or slot_mapping.numel() != int(siblings) * mk.shape[2]:
        raise ValueError("delta must hold one shift per sibling and slot_mapping one slot per "
                         "(sibling, token)")
    ek, ev = (k_list[2].shape[0], v_list[2].shape[0]) if entries is None else entries
    _check(lib.kvfix_diff_restore_split(_ptr(mk), _ptr(mv), plane_desc(mk), _ptr(k_list[0]), _ptr(v_list[0]),
                                        _ptr(k_list[1]), _ptr(v_list[1]), _ptr(k_list[2]), _ptr(v_list[2]),
                                        int(ek), int(ev), int(siblings), int(block_tokens), _ptr(delta),
                                        float(rope_base), _ptr(slot_mapping), _ptr(pool_k), _ptr(pool_v),
                                        plane_desc(pool_k.unsqueeze(0)), _stream(mk)))
    return pool_k, pool_v


def selftest_wait(limit_cycles: int, flag=None):
    """Launch the bounded-wait self test on the current stream (see kvfix_selftest_wait)."""
    if flag is not None:
        _i32(flag, "flag")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _check(lib.kvfix_selftest_wait(int(limit_cycles), _ptr(flag), s))


def anchor_gate_correct(k_src, v_src, factors: dict, prefix: int, delta, rope_base: float,
                        temperature: float = 1.0, tau: float = 0.5, out_k=None, out_v=None):
    """The gate and the correction in one pass (see kvfix_anchor_gate_correct).  Returns
    (out_k, out_v, w_k, w_v, d, g, hbar, accept)."""
    _bf16(k_src, "k_src")
    _bf16(v_src, "v_src")
    _i32(delta, "delta")
    C, L, n, H, Dh = k_src.shape
    V, r = factors["a_c_k"].shape[1], factors["a_c_k"].shape[-1]
    names = ("a_c_k", "b_ct_k", "a_c_v", "b_ct_v", "a_d_k", "b_dt_k", "a_d_v", "b_dt_v")
    for nm in names:
        _factor(factors[nm], nm, (C, V, L, n, r) if nm.startswith("a_") else (C, V, L, H * Dh, r))
    dev = k_src.device
    out_k = torch.empty_like(k_src) if out_k is None else out_k
    out_v = torch.empty_like(v_src) if out_v is None else out_v
    w_k = torch.empty((C, L, n, V), dtype=torch.float32, device=dev)
    w_v = torch.empty_like(w_k)
    d = torch.empty((C, V), dtype=torch.float64, device=dev)
    g = torch.empty_like(d)
    hbar = torch.empty(C, dtype=torch.float64, device=dev)
    acc = torch.empty(C, dtype=torch.int32, device=dev)
    desc = plane_desc(k_src)
    nbytes = lib.kvfix_anchor_gate_workspace_bytes(desc, V, n)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _check(lib.kvfix_anchor_gate_correct(_ptr(k_src), _ptr(v_src), desc, *[_ptr(factors[nm]) for nm in names], V, r,
                                         int(prefix), float(temperature), float(tau), _ptr(delta), float(rope_base),
                                         _ptr(d), _ptr(g), _ptr(hbar), _ptr(acc), _ptr(w_k), _ptr(w_v), _ptr(out_k),
                                         _ptr(out_v), plane_desc(out_k), _ptr(ws), ws.numel(), _stream(k_src)))
    return out_k, out_v, w_k, w_v, d, g, hbar, acc
