"""Storage accounting for the two ways of keeping many agents' KV caches: the anchor pool
and the master-mirror layout.  Plain host arithmetic, no device work.

KVCMAS: Efficient KV cache Correction for Shared Context in Multi-Agent Systems, section
3.1: each anchor keeps a full-dimensional base cache and one correction per consuming
agent, so a pool of V anchors serving N agents holds V (1 + N) caches -- O(V N L D) per
pool; section 3.3 (Eq. 7) stores each of those states as two rank-r factors per layer and
plane instead.

TokenDance: Scaling Multi-Agent LLM Serving via Collective KV Cache Sharing, section 6.4
(the implied capacity gain): with a master and N - 1 mirrors stored
as diffs compressed R-fold, a round of N agents costs about 1 + (N - 1) / R full caches
instead of N.
"""
from __future__ import annotations

BF16_BYTES = 2


def kv_cache_bytes(layers: int, tokens: int, kv_heads: int, head_dim: int, elem_bytes: int = BF16_BYTES) -> int:
    """Bytes of one full cache, keys and values, every layer."""
    return 2 * layers * tokens * kv_heads * head_dim * elem_bytes


def anchor_state_bytes(layers: int, tokens: int, kv_heads: int, head_dim: int, rank: int | None = None,
                       elem_bytes: int = BF16_BYTES) -> int:
    """Bytes of one anchor state (a base cache or one agent's correction): the full cache,
    or with `rank` the two factors per layer and plane -- A [tokens x r] and Bt
    [kv_heads*head_dim x r]."""
    if rank is None:
        return kv_cache_bytes(layers, tokens, kv_heads, head_dim, elem_bytes)
    return 2 * layers * (tokens + kv_heads * head_dim) * rank * elem_bytes


def anchor_pool_bytes(layers: int, tokens: int, kv_heads: int, head_dim: int, anchors: int, agents: int,
                      rank: int | None = None, elem_bytes: int = BF16_BYTES) -> dict:
    """Bytes of an anchor pool of `anchors` entries, each with a base state and one
    correction per agent.  Returns {"bases", "corrections", "total"}."""
    one = anchor_state_bytes(layers, tokens, kv_heads, head_dim, rank, elem_bytes)
    bases = anchors * one
    corrections = anchors * agents * one
    return {"bases": bases, "corrections": corrections, "total": bases + corrections}


def mirror_round_copies(agents: int, compression: float) -> float:
    """Full caches a round of `agents` costs under the master-mirror layout: one master
    plus agents - 1 mirrors, each 1/compression of a full cache."""
    if agents < 1 or compression <= 0:
        raise ValueError("agents must be >= 1 and compression > 0")
    return 1.0 + (agents - 1) / compression


def mirror_memory_reduction(agents: int, compression: float) -> float:
    """How many times less KV memory a round takes than `agents` dense caches."""
    return agents / mirror_round_copies(agents, compression)


def diff_stored_bytes(siblings: int, layers: int, tokens: int, kv_heads: int, head_dim: int, block_tokens: int,
                      entries: int, planes_per_entry: int = 2, lists: int = 1,
                      elem_bytes: int = BF16_BYTES) -> int:
    """Bytes the block-sparse diffs of `siblings` take: the packed payload (`entries`
    blocks of `planes_per_entry` planes), plus per list the dirty-block bit mask (whole
    32-bit words) and the int64 offsets (one per block and one total)."""
    blocks = siblings * layers * (tokens // block_tokens)
    payload = entries * planes_per_entry * block_tokens * kv_heads * head_dim * elem_bytes
    index = lists * (4 * ((blocks + 31) // 32) + 8 * (blocks + 1))
    return payload + index


def diff_compression(siblings: int, layers: int, tokens: int, kv_heads: int, head_dim: int, block_tokens: int,
                     entries: int, elem_bytes: int = BF16_BYTES) -> float:
    """Dense bytes of the siblings divided by the bytes of their joint diffs."""
    dense = siblings * kv_cache_bytes(layers, tokens, kv_heads, head_dim, elem_bytes)
    return dense / diff_stored_bytes(siblings, layers, tokens, kv_heads, head_dim, block_tokens, entries,
                                     elem_bytes=elem_bytes)
