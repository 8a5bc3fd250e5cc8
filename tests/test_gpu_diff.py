"""GPU parity of the block-sparse sibling diff (encode and gather): bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from cross_context_kv_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def kvfix():
    from cross_context_kv_gb300 import kvfix as k
    return k


SMALL_DIFF = [
    synth.SIBLINGS_8B.with_(name="diff_small", siblings=5, layers=3, tokens=96, kv_heads=2, head_dim=64, seed=50),
    synth.SIBLINGS_8B.with_(name="diff_odd_blocks", siblings=3, layers=2, tokens=320, kv_heads=1,
                            head_dim=128, block_tokens=32, frac_lo=0.2, frac_hi=0.5, seed=51),
]


def _encode_check(cfg, inp):
    mask, offsets, payload, entries = kvfix().diff_encode(inp["master_k"], inp["master_v"], inp["sib_k"],
                                                          inp["sib_v"], cfg.block_tokens)
    kvfix().check_status()
    omask, ooffs, opay, ototal = oracle.diff_encode(synth.bits(inp["master_k"]), synth.bits(inp["master_v"]),
                                                    synth.bits(inp["sib_k"]), synth.bits(inp["sib_v"]),
                                                    cfg.block_tokens)
    assert entries == ototal
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), omask)
    assert np.array_equal(offsets.cpu().numpy(), ooffs)
    assert np.array_equal(synth.bits(payload[:entries]), opay)
    return mask, offsets, payload, entries


@pytest.mark.parametrize("cfg", SMALL_DIFF, ids=lambda c: c.name)
def test_diff_encode_gather_bit_exact(cfg):
    inp = synth.diff_inputs(cfg, DEV)
    mask, offsets, payload, entries = _encode_check(cfg, inp)
    ok, ov = kvfix().diff_gather(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                                 cfg.block_tokens, payload_entries=entries)
    kvfix().check_status()
    assert torch.equal(ok.view(torch.int16), inp["sib_k"].view(torch.int16))
    assert torch.equal(ov.view(torch.int16), inp["sib_v"].view(torch.int16))


def test_diff_identical_siblings_and_single_word():
    cfg = SMALL_DIFF[0]
    inp = synth.diff_inputs(cfg, DEV)
    same_k = inp["master_k"].unsqueeze(0).repeat(4, 1, 1, 1, 1)
    same_v = inp["master_v"].unsqueeze(0).repeat(4, 1, 1, 1, 1)
    mask, offsets, payload, entries = kvfix().diff_encode(inp["master_k"], inp["master_v"], same_k, same_v, 16)
    assert entries == 0 and not mask.any() and not offsets.any()
    # flip the sign of one zero: -0 and +0 are different words
    same_k[2, 1, 37, 1, 5] = 0.0
    mk = inp["master_k"].clone()
    mk[1, 37, 1, 5] = -0.0
    mask, offsets, payload, entries = kvfix().diff_encode(mk, inp["master_v"], same_k, same_v, 16)
    L, nblk = cfg.layers, cfg.tokens // 16
    dirty = [i for i in range(4 * L * nblk) if (mask.cpu().numpy().view(np.uint32)[i // 32] >> (i % 32)) & 1]
    changed = {(2 * L + 1) * nblk + 37 // 16}
    others = {(s * L + 1) * nblk + 37 // 16 for s in range(4)}  # every sibling now differs from mk there
    assert set(dirty) == others | changed


def test_diff_capacity_too_small():
    cfg = SMALL_DIFF[0]
    inp = synth.diff_inputs(cfg, DEV)
    _, _, _, total = kvfix().diff_encode(inp["master_k"], inp["master_v"], inp["sib_k"], inp["sib_v"], 16)
    with pytest.raises(kvfix().KvfixError) as e:
        kvfix().diff_encode(inp["master_k"], inp["master_v"], inp["sib_k"], inp["sib_v"], 16, capacity=total - 1)
    assert e.value.status == kvfix().ENOSPACE
    # asynchronous form: entries beyond the capacity are skipped and flagged
    kvfix().diff_encode(inp["master_k"], inp["master_v"], inp["sib_k"], inp["sib_v"], 16, capacity=total - 1,
                        sync=False)
    with pytest.raises(kvfix().KvfixError) as e:
        kvfix().check_status()
    assert e.value.status == kvfix().ENOSPACE


@pytest.mark.slow
def test_full_size_diff_bit_exact():
    """16 siblings at 8B shape, the benchmark's launch configuration: every mask bit,
    offset and payload word equals the oracle's, and gather restores every sibling."""
    cfg = synth.SIBLINGS_8B
    inp = synth.diff_inputs(cfg, DEV)
    mask, offsets, payload, entries = _encode_check(cfg, inp)
    ok, ov = kvfix().diff_gather(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                                 cfg.block_tokens, payload_entries=entries)
    kvfix().check_status()
    assert torch.equal(ok.view(torch.int16), inp["sib_k"].view(torch.int16))
    assert torch.equal(ov.view(torch.int16), inp["sib_v"].view(torch.int16))
    full = 2 * inp["sib_k"].numel() * 2
    stored = entries * 2 * cfg.block_tokens * cfg.kv_heads * cfg.head_dim * 2 + mask.numel() * 4 + offsets.numel() * 8
    print(f"siblings_8b: {entries} dirty entries, compression {full / stored:.1f}x")


# ------------------------------------------------------------ fused diff restore

def _restore_setup(cfg, skip=0.1, spare_pages=3):
    inp = synth.diff_inputs(cfg, DEV)
    mask, offsets, payload, entries = kvfix().diff_encode(inp["master_k"], inp["master_v"], inp["sib_k"],
                                                          inp["sib_v"], cfg.block_tokens)
    tgt = synth.restore_inputs(cfg, DEV, skip=skip, spare_pages=spare_pages)
    shape = (cfg.layers, tgt["slots"], cfg.kv_heads, cfg.head_dim)
    g = torch.Generator(device=DEV).manual_seed(cfg.seed + 7)
    pool0 = torch.randn(shape, generator=g, device=DEV).to(torch.bfloat16)  # rows not restored keep this
    return inp, (mask, offsets, payload, entries), tgt, pool0


def _assert_k_rotation_close(got, ref, src, delta, base, what):
    """fp32 rotation against the oracle's fp64 one: within the K tolerance, at most 1e-3 of
    the words differ from the oracle's, and every word lies within half a bf16 unit of the
    exact rotation plus a float32 bound on the computation (2^-20 (|x_i| + |x_{i+D/2}|))."""
    from helpers import assert_close_kv
    assert_close_kv(got, ref, what)
    ne = got != ref
    assert ne.mean() < 1e-3, f"{what}: {ne.mean():.2e} of the words differ"
    x = oracle.bf16_decode(src)
    exact = oracle.rotate_f64(x, float(delta), base)
    D = x.shape[-1]
    mag = np.abs(x[..., : D // 2]) + np.abs(x[..., D // 2:])
    mag = np.concatenate([mag, mag], -1)
    y = oracle.bf16_decode(got)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(y), 1e-38))) - 7)
    assert (np.abs(y - exact) <= 0.5 * ulp + 2.0 ** -20 * mag).all(), f"{what}: a word is outside the bound"


@pytest.mark.parametrize("cfg", SMALL_DIFF, ids=lambda c: c.name)
def test_diff_restore_matches_oracle(cfg):
    inp, (mask, offsets, payload, entries), tgt, pool0 = _restore_setup(cfg)
    pk, pv = pool0.clone(), pool0.clone()
    kvfix().diff_restore(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                         cfg.block_tokens, tgt["delta"], cfg.rope_base, tgt["slot_mapping"], pk, pv,
                         payload_entries=entries)
    kvfix().check_status()
    ok, ov = oracle.diff_restore(synth.bits(inp["master_k"]), synth.bits(inp["master_v"]),
                                 mask.cpu().numpy().view(np.uint32), offsets.cpu().numpy(),
                                 synth.bits(payload[:max(entries, 1)]), cfg.siblings, cfg.block_tokens,
                                 tgt["delta"].cpu().numpy(), cfg.rope_base,
                                 tgt["slot_mapping"].cpu().numpy(), synth.bits(pool0), synth.bits(pool0))
    assert np.array_equal(synth.bits(pv), ov)
    gk = synth.bits(pk)
    smap = tgt["slot_mapping"].cpu().numpy()
    delta = tgt["delta"].cpu().numpy()
    exact = np.ones(tgt["slots"], bool)      # unrestored rows and rows of unshifted siblings
    sib_k = synth.bits(inp["sib_k"])
    for s in range(cfg.siblings):
        if delta[s] != 0:
            on = smap[s] >= 0
            exact[smap[s][on]] = False
            _assert_k_rotation_close(gk[:, smap[s][on]], ok[:, smap[s][on]], sib_k[s][:, on], delta[s],
                                     cfg.rope_base, f"{cfg.name} sibling {s}")
    assert (smap < 0).any() and (delta == 0).any() and (delta != 0).any()
    assert np.array_equal(gk[:, exact], ok[:, exact])


@pytest.mark.parametrize("cfg", SMALL_DIFF, ids=lambda c: c.name)
def test_diff_restore_equals_rerope_of_gather(cfg):
    """Restore fuses gather, rerope and the slot scatter: the same words as those three
    kernels run one after another."""
    inp, (mask, offsets, payload, entries), tgt, pool0 = _restore_setup(cfg, skip=0.0, spare_pages=0)
    pk, pv = pool0.clone(), pool0.clone()
    kvfix().diff_restore(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                         cfg.block_tokens, tgt["delta"], cfg.rope_base, tgt["slot_mapping"], pk, pv,
                         payload_entries=entries)
    gk, gv = kvfix().diff_gather(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                                 cfg.block_tokens, payload_entries=entries)
    rk = kvfix().rerope(gk, tgt["delta"], cfg.rope_base)
    kvfix().check_status()
    slot = tgt["slot_mapping"].long()
    for s in range(cfg.siblings):
        assert torch.equal(pk[:, slot[s]].view(torch.int16), rk[s].view(torch.int16))
        assert torch.equal(pv[:, slot[s]].view(torch.int16), inp["sib_v"][s].view(torch.int16))


def test_diff_restore_out_of_range_slot_is_flagged_and_skipped():
    cfg = SMALL_DIFF[0]
    inp, (mask, offsets, payload, entries), tgt, pool0 = _restore_setup(cfg, skip=0.0, spare_pages=0)
    smap = tgt["slot_mapping"].clone()
    smap[1, 5] = tgt["slots"]
    pk, pv = pool0.clone(), pool0.clone()
    kvfix().diff_restore(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                         cfg.block_tokens, tgt["delta"], cfg.rope_base, smap, pk, pv, payload_entries=entries)
    with pytest.raises(kvfix().KvfixError) as e:
        kvfix().check_status()
    assert e.value.status == kvfix().EDEVICE
    missed = int(tgt["slot_mapping"][1, 5])
    assert torch.equal(pk[:, missed].view(torch.int16), pool0[:, missed].view(torch.int16))
    assert torch.equal(pv[:, missed].view(torch.int16), pool0[:, missed].view(torch.int16))


@pytest.mark.slow
def test_full_size_diff_restore():
    """16 siblings at 8B shape into a paged pool, the benchmark's launch configuration:
    every row equals the gather + rerope composition bit for bit, and sampled rows match
    the oracle's rotation of the synthetic siblings."""
    cfg = synth.SIBLINGS_8B
    inp = synth.diff_inputs(cfg, DEV)
    mask, offsets, payload, entries = kvfix().diff_encode(inp["master_k"], inp["master_v"], inp["sib_k"],
                                                          inp["sib_v"], cfg.block_tokens)
    tgt = synth.restore_inputs(cfg, DEV)
    shape = (cfg.layers, tgt["slots"], cfg.kv_heads, cfg.head_dim)
    pk = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    pv = torch.empty_like(pk)
    kvfix().diff_restore(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                         cfg.block_tokens, tgt["delta"], cfg.rope_base, tgt["slot_mapping"], pk, pv,
                         payload_entries=entries)
    kvfix().check_status()
    slot = tgt["slot_mapping"].long()
    delta_h = tgt["delta"].cpu().numpy()
    rng = np.random.default_rng(5)
    for s in range(cfg.siblings):
        rk = kvfix().rerope(inp["sib_k"][s:s + 1], tgt["delta"][s:s + 1], cfg.rope_base)
        assert torch.equal(pk[:, slot[s]].view(torch.int16), rk[0].view(torch.int16))
        assert torch.equal(pv[:, slot[s]].view(torch.int16), inp["sib_v"][s].view(torch.int16))
        del rk
        ts = np.sort(rng.choice(cfg.tokens, 24, replace=False))
        sib = synth.bits(inp["sib_k"][s][:, ts])                      # [L][24][H][D]
        ref = oracle.rerope(sib[None], delta_h[s:s + 1], cfg.rope_base)[0]
        got = synth.bits(pk[:, slot[s, torch.as_tensor(ts, device=DEV)]])
        if delta_h[s] == 0:
            assert np.array_equal(got, sib)
        else:
            _assert_k_rotation_close(got, ref, sib, delta_h[s], cfg.rope_base, f"sibling {s}")


# ------------------------------------------------------------ per-plane lists, master

def _planes_differ(inp, cfg, seed):
    """Make the K and V planes touch different blocks: flip V words in extra blocks and
    restore K in some of the dirty ones."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    S, L, n = cfg.siblings, cfg.layers, cfg.tokens
    bt = cfg.block_tokens
    sk, sv = inp["sib_k"], inp["sib_v"]
    for s in range(S):
        for _ in range(3):
            l = int(torch.randint(L, (1,), generator=g))
            t = int(torch.randint(n, (1,), generator=g))
            sv[s, l, t, 0, 0] = -sv[s, l, t, 0, 0] + 1.0
        blocks = inp["dirty_blocks"][s]
        if len(blocks):
            b = int(blocks[0])
            sk[s, :, b * bt:(b + 1) * bt] = inp["master_k"][:, b * bt:(b + 1) * bt]


def _split_check(cfg, inp):
    kl, vl, ent = kvfix().diff_encode_split(inp["master_k"], inp["master_v"], inp["sib_k"], inp["sib_v"],
                                            cfg.block_tokens)
    kvfix().check_status()
    okd, ovd = oracle.diff_encode_split(synth.bits(inp["master_k"]), synth.bits(inp["master_v"]),
                                        synth.bits(inp["sib_k"]), synth.bits(inp["sib_v"]), cfg.block_tokens)
    for got, ref, e in ((kl, okd, ent[0]), (vl, ovd, ent[1])):
        assert e == ref[1][-1]
        assert np.array_equal(got[0].cpu().numpy().view(np.uint32), ref[0])
        assert np.array_equal(got[1].cpu().numpy(), ref[1])
        assert np.array_equal(synth.bits(got[2][:e]), ref[2])
    ok, ov = kvfix().diff_gather_split(inp["master_k"], inp["master_v"], kl, vl, cfg.siblings, cfg.block_tokens,
                                       entries=ent)
    kvfix().check_status()
    assert torch.equal(ok.view(torch.int16), inp["sib_k"].view(torch.int16))
    assert torch.equal(ov.view(torch.int16), inp["sib_v"].view(torch.int16))
    return kl, vl, ent


@pytest.mark.parametrize("cfg", SMALL_DIFF, ids=lambda c: c.name)
def test_split_diff_bit_exact(cfg):
    inp = synth.diff_inputs(cfg, DEV)
    kl, vl, _ = _split_check(cfg, inp)
    # the generator dirties K and V in the same blocks: the two lists coincide
    assert torch.equal(kl[0], vl[0]) and torch.equal(kl[1], vl[1])
    _planes_differ(inp, cfg, 5)
    kl, vl, ent = _split_check(cfg, inp)
    assert not torch.equal(kl[0], vl[0])


@pytest.mark.parametrize("cfg", SMALL_DIFF, ids=lambda c: c.name)
def test_split_restore_equals_joint_restore(cfg):
    """The restore from per-plane lists writes the joint restore's words, also where the K
    and V planes of a sibling are dirty in different blocks; V rows equal the oracle's."""
    inp = synth.diff_inputs(cfg, DEV)
    _planes_differ(inp, cfg, 8)
    kl, vl, ent = _split_check(cfg, inp)
    mask, offsets, payload, entries = kvfix().diff_encode(inp["master_k"], inp["master_v"], inp["sib_k"],
                                                          inp["sib_v"], cfg.block_tokens)
    tgt = synth.restore_inputs(cfg, DEV, skip=0.1, spare_pages=3)
    shape = (cfg.layers, tgt["slots"], cfg.kv_heads, cfg.head_dim)
    g = torch.Generator(device=DEV).manual_seed(cfg.seed + 9)
    pool0 = torch.randn(shape, generator=g, device=DEV).to(torch.bfloat16)
    jk, jv = pool0.clone(), pool0.clone()
    kvfix().diff_restore(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                         cfg.block_tokens, tgt["delta"], cfg.rope_base, tgt["slot_mapping"], jk, jv,
                         payload_entries=entries)
    sk, sv = pool0.clone(), pool0.clone()
    kvfix().diff_restore_split(inp["master_k"], inp["master_v"], kl, vl, cfg.siblings, cfg.block_tokens,
                               tgt["delta"], cfg.rope_base, tgt["slot_mapping"], sk, sv, entries=ent)
    kvfix().check_status()
    assert torch.equal(sk.view(torch.int16), jk.view(torch.int16))
    assert torch.equal(sv.view(torch.int16), jv.view(torch.int16))
    _, ov = oracle.diff_restore(synth.bits(inp["master_k"]), synth.bits(inp["master_v"]),
                                mask.cpu().numpy().view(np.uint32), offsets.cpu().numpy(),
                                synth.bits(payload[:max(entries, 1)]), cfg.siblings, cfg.block_tokens,
                                tgt["delta"].cpu().numpy(), cfg.rope_base,
                                tgt["slot_mapping"].cpu().numpy(), synth.bits(pool0), synth.bits(pool0))
    assert np.array_equal(synth.bits(sv), ov)


def test_split_restore_with_empty_lists_and_one_dirty_plane():
    """Siblings equal to the master give two empty lists: every restored row is the master's
    (keys re-aligned).  Then one value word changes in one sibling: only the value list
    holds an entry, and the restore still equals the joint one."""
    cfg = SMALL_DIFF[0]
    inp = synth.diff_inputs(cfg, DEV)
    S = cfg.siblings
    sk = inp["master_k"].unsqueeze(0).repeat(S, 1, 1, 1, 1)
    sv = inp["master_v"].unsqueeze(0).repeat(S, 1, 1, 1, 1)
    tgt = synth.restore_inputs(cfg, DEV, skip=0.0, spare_pages=2)
    shape = (cfg.layers, tgt["slots"], cfg.kv_heads, cfg.head_dim)
    for step in range(2):
        if step == 1:
            sv[2, 1, 40, 0, 3] = sv[2, 1, 40, 0, 3] + 1.0
        kl, vl, ent = kvfix().diff_encode_split(inp["master_k"], inp["master_v"], sk, sv, cfg.block_tokens)
        mask, offsets, payload, entries = kvfix().diff_encode(inp["master_k"], inp["master_v"], sk, sv,
                                                              cfg.block_tokens)
        kvfix().check_status()
        assert ent == ((0, 0) if step == 0 else (0, 1)) and entries == step
        jk, jv = torch.zeros(shape, dtype=torch.bfloat16, device=DEV), torch.zeros(shape, dtype=torch.bfloat16, device=DEV)
        pk, pv = torch.zeros_like(jk), torch.zeros_like(jv)
        kvfix().diff_restore(inp["master_k"], inp["master_v"], mask, offsets, payload, S, cfg.block_tokens,
                             tgt["delta"], cfg.rope_base, tgt["slot_mapping"], jk, jv, payload_entries=entries)
        kvfix().diff_restore_split(inp["master_k"], inp["master_v"], kl, vl, S, cfg.block_tokens, tgt["delta"],
                                   cfg.rope_base, tgt["slot_mapping"], pk, pv, entries=ent)
        kvfix().check_status()
        assert torch.equal(pk.view(torch.int16), jk.view(torch.int16))
        assert torch.equal(pv.view(torch.int16), jv.view(torch.int16))
        slot = tgt["slot_mapping"].long()
        for s in range(S):
            rk = kvfix().rerope(inp["master_k"].unsqueeze(0), tgt["delta"][s:s + 1], cfg.rope_base)
            assert torch.equal(pk[:, slot[s]].view(torch.int16), rk[0].view(torch.int16))
            assert torch.equal(pv[:, slot[s]].view(torch.int16), sv[s].view(torch.int16))


@pytest.mark.slow
def test_full_size_split_diff():
    cfg = synth.SIBLINGS_8B
    inp = synth.diff_inputs(cfg, DEV)
    _planes_differ(inp, cfg, 6)
    kl, vl, ent = kvfix().diff_encode_split(inp["master_k"], inp["master_v"], inp["sib_k"], inp["sib_v"],
                                            cfg.block_tokens)
    mask, offsets, payload, entries = kvfix().diff_encode(inp["master_k"], inp["master_v"], inp["sib_k"],
                                                          inp["sib_v"], cfg.block_tokens)
    kvfix().check_status()
    assert torch.equal(kl[0] | vl[0], mask)
    assert max(ent) <= entries <= ent[0] + ent[1]
    ok, ov = kvfix().diff_gather_split(inp["master_k"], inp["master_v"], kl, vl, cfg.siblings, cfg.block_tokens,
                                       entries=ent)
    kvfix().check_status()
    assert torch.equal(ok.view(torch.int16), inp["sib_k"].view(torch.int16))
    assert torch.equal(ov.view(torch.int16), inp["sib_v"].view(torch.int16))
    del ok, ov
    tgt = synth.restore_inputs(cfg, DEV)
    shape = (cfg.layers, tgt["slots"], cfg.kv_heads, cfg.head_dim)
    jk = torch.zeros(shape, dtype=torch.bfloat16, device=DEV)
    jv, sk, sv = torch.zeros_like(jk), torch.zeros_like(jk), torch.zeros_like(jk)
    kvfix().diff_restore(inp["master_k"], inp["master_v"], mask, offsets, payload, cfg.siblings,
                         cfg.block_tokens, tgt["delta"], cfg.rope_base, tgt["slot_mapping"], jk, jv,
                         payload_entries=entries)
    kvfix().diff_restore_split(inp["master_k"], inp["master_v"], kl, vl, cfg.siblings, cfg.block_tokens,
                               tgt["delta"], cfg.rope_base, tgt["slot_mapping"], sk, sv, entries=ent)
    kvfix().check_status()
    assert torch.equal(sk.view(torch.int16), jk.view(torch.int16))
    assert torch.equal(sv.view(torch.int16), jv.view(torch.int16))


def test_master_select_matches_oracle():
    rng = np.random.default_rng(80)
    for A, R, n in ((8, 8, 512), (3, 1, 4096), (16, 2, 1000)):
        dk = rng.random((A * R, n)).astype(np.float32)
        dv = rng.random((A * R, n)).astype(np.float32)
        m, tot = kvfix().master_select(torch.as_tensor(dk, device=DEV), torch.as_tensor(dv, device=DEV), A)
        rm, rtot = oracle.master_select(dk, dv, A)
        np.testing.assert_allclose(tot.cpu().numpy(), rtot, rtol=1e-12)
        srt = np.sort(rtot)
        if (srt[1] - srt[0]) / srt[1] > 1e-12:
            assert int(m.item()) == rm
        mk, _ = kvfix().master_select(torch.as_tensor(dk, device=DEV), None, A)
        assert int(mk.item()) == oracle.master_select(dk, None, A)[0]
    same = torch.as_tensor(np.tile(dk[:2], (16, 1)), device=DEV)
    assert int(kvfix().master_select(same, same, 16)[0].item()) == 0


def test_bounded_wait_times_out_and_the_context_survives():
    """The pipelines' bounded wait, run out on purpose (a barrier phase nothing completes,
    a flag nothing sets): the status word reports a timeout, reading it clears it, and
    the next calls run normally."""
    kvfix().check_status()
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvfix().selftest_wait(2_000_000, flag)
    with pytest.raises(kvfix().KvfixError) as e:
        kvfix().check_status()
    assert e.value.status == kvfix().ETIMEOUT
    kvfix().check_status()                       # cleared
    k = torch.randn((1, 2, 64, 2, 64), device=DEV).to(torch.bfloat16)
    out = kvfix().rerope(k, torch.zeros(1, dtype=torch.int32, device=DEV), 1e4)
    kvfix().check_status()
    assert torch.equal(out.view(torch.int16), k.view(torch.int16))
