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
