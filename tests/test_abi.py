"""The C ABI: the library builds, loads and exports every entry point include/kvfix.h
declares; host-side argument checks reject bad calls before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvfix.h")


@pytest.fixture(scope="module")
def lib():
    from cross_context_kv_gb300 import build
    build.build()
    from cross_context_kv_gb300 import kvfix
    return kvfix


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"KVFIX_API\s+[\w\s\*]+?\b(kvfix_\w+)\s*\(", text)


def test_header_declares_the_seven_calls_and_the_restore():
    names = set(declared_symbols())
    for call in ("kvfix_rerope", "kvfix_score_topk", "kvfix_draft_rank", "kvfix_mean_correct",
                 "kvfix_lowrank_apply", "kvfix_diff_encode", "kvfix_diff_gather", "kvfix_diff_restore"):
        assert call in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_symbols() if not hasattr(raw, n)]
    assert not missing, missing
    assert set(declared_symbols()) == set(lib.SIGNATURES), "binding signatures out of sync with the header"


def test_binding_argument_counts_match_header(lib):
    text = open(HEADER).read()
    for name in declared_symbols():
        m = re.search(r"KVFIX_API[^;(]*\b" + name + r"\s*\(([^)]*)\)", text)
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(lib.SIGNATURES[name][1]), name


def _desc(lib, C=1, L=1, n=16, H=1, D=64):
    row = H * D
    return lib.KvDesc(C, L, n, H, D, L * n * row, n * row, row)


def test_host_validation_rejects_bad_arguments(lib):
    L = lib.lib
    fake = ctypes.c_void_p(1 << 20)      # never dereferenced: the checks fail first
    odd = ctypes.c_void_p((1 << 20) + 2)  # not 16-byte aligned
    bad_dim = _desc(lib, D=24)
    assert L.kvfix_rerope(fake, bad_dim, fake, bad_dim, fake, 1e4, None) == lib.EINVAL
    assert b"head_dim" in L.kvfix_last_error()
    assert L.kvfix_rerope(odd, _desc(lib), fake, _desc(lib), fake, 1e4, None) == lib.EINVAL
    assert L.kvfix_rerope(fake, _desc(lib), fake, _desc(lib), fake, 0.5, None) == lib.EINVAL
    assert L.kvfix_rerope(None, _desc(lib), fake, _desc(lib), fake, 1e4, None) == lib.EINVAL
    # partial overlap of input and output is refused
    assert L.kvfix_rerope(fake, _desc(lib), ctypes.c_void_p((1 << 20) + 64), _desc(lib), fake, 1e4,
                          None) == lib.EINVAL
    d = _desc(lib)
    # b out of range
    assert L.kvfix_score_topk(fake, fake, d, fake, fake, d, 1, fake, 1e4, 17, fake, fake, fake, fake,
                              fake, fake, None, None, None, None) == lib.EINVAL
    # fresh chunks != agents * reuse chunks
    assert L.kvfix_score_topk(fake, fake, d, fake, fake, d, 2, fake, 1e4, 3, fake, fake, fake, fake,
                              fake, fake, None, None, None, None) == lib.EINVAL
    # rank not a multiple of 16
    assert L.kvfix_lowrank_apply(fake, _desc(lib, D=128), fake, fake, 8, ctypes.c_void_p(1 << 30),
                                 _desc(lib, D=128), None) == lib.EINVAL
    # block size must divide the tokens
    dm = _desc(lib, n=40)
    assert L.kvfix_diff_encode(fake, fake, dm, fake, fake, dm, 16, fake, fake, fake, 10, None, None) == lib.EINVAL
    # workspace too small
    dk = _desc(lib, C=1, L=2, n=64, H=1, D=128)
    need = L.kvfix_draft_rank_workspace_bytes(dk, 1)
    assert need > 0
    assert L.kvfix_draft_rank(fake, dk, fake, 2, 8, 1, 4, fake, fake, None, None, dk, None, None,
                              fake, need - 16, None) == lib.EINVAL
    # grouped queries beyond 16 rows per KV head
    assert L.kvfix_draft_rank(fake, dk, fake, 3, 8, 1, 4, fake, fake, None, None, dk, None, None,
                              fake, need, None) == lib.EINVAL
    # restore: the pool must match the master's layers and lie apart from it
    dm, far = _desc(lib, L=2, n=32), ctypes.c_void_p(1 << 30)
    far_v = ctypes.c_void_p((1 << 30) + (1 << 24))
    pool = _desc(lib, L=2, n=100)
    assert L.kvfix_diff_restore(fake, fake, dm, fake, fake, None, 0, 2, 16, fake, 1e4, fake, far, far_v,
                                _desc(lib, L=3, n=100), None) == lib.EINVAL
    assert b"layers" in L.kvfix_last_error()
    assert L.kvfix_diff_restore(fake, fake, dm, fake, fake, None, 0, 2, 16, fake, 1e4, fake, fake, far_v,
                                pool, None) == lib.EINVAL
    assert L.kvfix_diff_restore(fake, fake, dm, fake, fake, None, 0, 2, 16, None, 1e4, fake, far, far_v,
                                pool, None) == lib.EINVAL
    assert L.kvfix_diff_restore(fake, fake, dm, fake, fake, None, 0, 2, 16, fake, 1.0, fake, far, far_v,
                                pool, None) == lib.EINVAL
    # the per-plane restore wants both lists and a valid pool like the joint one
    assert L.kvfix_diff_restore_split(fake, fake, dm, fake, None, fake, fake, None, None, 0, 0, 2, 16, fake, 1e4,
                                      fake, far, far_v, pool, None) == lib.EINVAL
    assert b"mask" in L.kvfix_last_error()
    assert L.kvfix_diff_restore_split(fake, fake, dm, fake, fake, fake, fake, None, None, 0, 3, 2, 16, fake, 1e4,
                                      fake, far, far_v, pool, None) == lib.EINVAL
    assert b"payload" in L.kvfix_last_error()
    assert L.kvfix_diff_restore_split(fake, fake, dm, fake, fake, fake, fake, None, None, 0, 0, 2, 16, fake, 1e4,
                                      fake, far, far_v, _desc(lib, L=3, n=100), None) == lib.EINVAL
    # repair layouts: tokens beyond 16384, an unknown layout, a budget above 1, max_rows too small
    assert L.kvfix_repair_layout(fake, 1, 16385, 0, 64, 1, 5, 0.25, 1, fake, 4000, fake, None) == lib.EINVAL
    assert L.kvfix_repair_layout(fake, 1, 1000, 3, 64, 1, 5, 0.25, 1, fake, 1000, fake, None) == lib.EINVAL
    assert L.kvfix_repair_layout(fake, 1, 1000, 2, 64, 6, 5, 0.25, 1, fake, 1000, fake, None) == lib.EINVAL
    assert L.kvfix_repair_layout(fake, 1, 1000, 2, 64, 1, 5, 0.25, 1, fake, 199, fake, None) == lib.EINVAL
    assert b"max_rows" in L.kvfix_last_error()
    assert L.kvfix_repair_layout(fake, 1, 1000, 1, 64, 1, 5, 0.25, 1, fake, 191, fake, None) == lib.EINVAL
    # row repair: a plane with io but no fresh pointer
    assert L.kvfix_repair_rows(fake, None, d, None, None, d, fake, 4, fake, None) == lib.EINVAL
    # master selection: no score plane
    assert L.kvfix_master_select(None, None, 4, 2, 16, fake, fake, None) == lib.EINVAL
    # per-plane diffs: a missing V mask
    assert L.kvfix_diff_encode_split(fake, fake, dm, fake, fake, dm, 16, fake, None, fake, fake, None, None, 0, 0,
                                     None, None) == lib.EINVAL
    assert L.kvfix_diff_gather_split(fake, fake, dm, fake, None, fake, fake, None, None, 0, 0, 1, 16, far, far_v,
                                     dm, None) == lib.EINVAL


def test_anchor_shared_memory_admission(lib):
    """Which (anchors, rank) the anchor kernels take: the resident first-factor tiles,
    row sums and rings must fit one SM's shared memory.  Ranks 16 and 32 take all 16
    anchors, rank 64 at most 8, for head_dim 64 and 128 alike.  A shape that fits gets
    past the shape check and fails the next host check instead (no GPU involved)."""
    L = lib.lib
    fake = ctypes.c_void_p(1 << 20)
    fake2 = ctypes.c_void_p(1 << 23)
    far, far_v = ctypes.c_void_p(1 << 30), ctypes.c_void_p((1 << 30) + (1 << 26))
    for H, D in ((8, 128), (2, 64)):
        src = _desc(lib, C=1, L=1, n=256, H=H, D=D)
        for rank in (16, 32, 64):
            for anchors in range(1, 17):
                fits = rank < 64 or anchors <= 8
                st = L.kvfix_anchor_correct(fake, fake2, src, *([fake] * 8), anchors, rank, 0.0, fake, 1e4, None,
                                            fake, fake2, far, far_v, src, None)
                msg = L.kvfix_last_error()
                assert st == lib.EINVAL
                assert (b"temperature" in msg) == fits and (b"shared memory" in msg) == (not fits), \
                    (H, D, rank, anchors, msg)
                st = L.kvfix_anchor_gate(fake, src, fake, fake, anchors, rank, 0, 1.0, 0.5, fake, fake, fake, fake,
                                         far, 1 << 20, None)
                msg = L.kvfix_last_error()
                assert st == lib.EINVAL
                assert (b"prefix" in msg) == fits and (b"shared memory" in msg) == (not fits), (rank, anchors, msg)


def test_version(lib):
    assert lib.version() == 100


def test_anchor_and_mean_correct_validation(lib):
    """The anchor and probe-mean calls reject bad arguments on the host, before any
    device work (no GPU needed: every case fails a check)."""
    L = lib.lib
    fake = ctypes.c_void_p(1 << 20)
    fake2 = ctypes.c_void_p(1 << 23)
    odd = ctypes.c_void_p((1 << 20) + 2)
    far, far_v = ctypes.c_void_p(1 << 30), ctypes.c_void_p((1 << 30) + (1 << 26))
    src = _desc(lib, C=2, L=2, n=256, H=8, D=128)
    f8 = [fake] * 8

    def correct(**kw):
        a = dict(k_src=fake, v_src=fake2, src=src, f=f8, anchors=10, rank=32, T=1.0, delta=fake, base=1e4,
                 accept=None, w_k=fake, w_v=fake2, k_out=far, v_out=far_v, out=src)
        a.update(kw)
        return L.kvfix_anchor_correct(a["k_src"], a["v_src"], a["src"], *a["f"], a["anchors"], a["rank"], a["T"],
                                      a["delta"], a["base"], a["accept"], a["w_k"], a["w_v"], a["k_out"],
                                      a["v_out"], a["out"], None)

    assert correct(rank=24) == lib.EINVAL and b"rank" in L.kvfix_last_error()
    assert correct(anchors=0) == lib.EINVAL and correct(anchors=17) == lib.EINVAL
    hd96 = _desc(lib, C=2, L=2, n=256, H=4, D=96)
    assert correct(src=hd96, out=hd96) == lib.EINVAL and b"head_dim" in L.kvfix_last_error()
    narrow = _desc(lib, C=2, L=2, n=256, H=1, D=64)   # a row of 64 features: not a whole chunk
    assert correct(src=narrow, out=narrow) == lib.EINVAL and b"multiple of 128" in L.kvfix_last_error()
    assert correct(base=1.0) == lib.EINVAL
    assert correct(T=0.0) == lib.EINVAL
    assert correct(w_k=None) == lib.EINVAL and b"required" in L.kvfix_last_error()
    assert correct(f=[fake] * 7 + [odd]) == lib.EINVAL and b"b_dt_v" in L.kvfix_last_error()
    # exactly in place is allowed; an output straddling the other plane's source is not
    assert correct(k_out=fake, v_out=ctypes.c_void_p((1 << 20) + 4096)) == lib.EINVAL
    assert b"overlap" in L.kvfix_last_error()

    need = L.kvfix_anchor_gate_workspace_bytes(src, 10, 256)
    assert need > 0 and L.kvfix_anchor_gate_workspace_bytes(src, 10, 128) <= need
    assert L.kvfix_anchor_gate_workspace_bytes(src, 0, 256) == 0

    def gate(**kw):
        a = dict(src=src, anchors=10, rank=32, prefix=256, T=1.0, tau=0.5, ws=far, ws_bytes=need)
        a.update(kw)
        return L.kvfix_anchor_gate(fake, a["src"], fake, fake, a["anchors"], a["rank"], a["prefix"], a["T"], a["tau"],
                                   fake, fake, fake, fake, a["ws"], a["ws_bytes"], None)

    assert gate(prefix=0) == lib.EINVAL and gate(prefix=257) == lib.EINVAL
    assert gate(tau=float("nan")) == lib.EINVAL
    assert gate(ws=None) == lib.EINVAL and b"workspace" in L.kvfix_last_error()
    assert gate(ws_bytes=need - 1) == lib.EINVAL
    assert gate(ws=ctypes.c_void_p((1 << 30) + 4)) == lib.EINVAL and b"aligned" in L.kvfix_last_error()

    # the one-pass call checks the gate's arguments too
    assert L.kvfix_anchor_gate_correct(fake, fake2, src, *f8, 10, 32, 256, 1.0, 0.5, fake, 1e4, fake, fake, fake,
                                       fake, fake, fake2, far, far_v, src, far, 0, None) == lib.EINVAL
    assert b"workspace" in L.kvfix_last_error()

    # probe-mean correction: b beyond the tokens, no agents, a plane without weights
    r = _desc(lib, C=1, L=2, n=64, H=2, D=64)
    args = [fake, fake2, r, far, far_v, r, ctypes.c_void_p(1 << 31), ctypes.c_void_p((1 << 31) + (1 << 26)), r]
    assert L.kvfix_mean_correct(*args, 1, fake, 1e4, fake, fake, 65, fake, fake, fake, fake, None) == lib.EINVAL
    assert L.kvfix_mean_correct(*args, 0, fake, 1e4, fake, fake, 8, fake, fake, fake, fake, None) == lib.EINVAL
    assert L.kvfix_mean_correct(*args, 1, fake, 1e4, fake, fake, 8, None, fake, fake, fake, None) == lib.EINVAL
    assert b"needs w" in L.kvfix_last_error()
    # the bounded-wait self test: a limit outside [1, 4e9]
    assert L.kvfix_selftest_wait(0, None, None) == lib.EINVAL
