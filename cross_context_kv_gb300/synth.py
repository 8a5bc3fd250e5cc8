"""Seeded synthetic workloads for the reused-KV-chunk repair path.

This module only DRAWS random tensors (torch generators, one stream per purpose so
that any slice can be regenerated on its own) and holds the workload shapes.  It
contains none of the repair arithmetic: no rotation, no scoring, no selection, no
correction.  The fresh key states of the repair workloads, which need a rotation,
are composed elsewhere from these draws (by the oracle in the tests, by the library
in the benchmark).

Draws depend on (seed, stream, device): a CUDA generator and a CPU generator give
different numbers for the same seed, so one run always draws on one device.

Workloads (synthetic stand-ins for the cache shapes the pages serve; no dataset,
no model weights):
  repair_tiny     2 layers, 4 KV heads x 64, one 256-token chunk, delta 137,
                  RoPE base 1e4, 5% heavy tokens ~ N(0,1), r = 0.1 (b = 26)
  repair_llama8b  32 layers, 8 x 128, one 4096-token chunk, delta ~ U{500..8000},
                  base 5e5, 3% heavy tokens ~ Student-t(3), r = 0.15 (b = 615)
  round_qwen14b   48 layers, 8 x 128, 8 agents x 8 shared 512-token blocks, agent
                  history ~ U{200..3000}, per-agent block permutation, base 1e6,
                  5% heavy ~ N(0,1), r = 0.1 (b = 52)
  siblings_8b     32 layers, 8 x 128, 8192 tokens, 16 siblings, 3-9% of 16-token
                  blocks redrawn as master + N(0, 0.2^2)
  lowrank_70b     80 layers, 8 KV / 64 query heads x 128, 4 chunks x 16384 tokens,
                  rank-16 A ~ N(0, 0.1^2), B ~ N(0,1), 2 draft queries ~ N(0,1),
                  fresh = reuse + N(0, 0.5^2), repair budget 819 rows per chunk
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import torch

BF16 = torch.bfloat16


# ----------------------------------------------------------------- configs

@dataclass(frozen=True)
class RepairConfig:
    """Chunk repair: re-rope + divergence + top-b + probe-mean correction."""
    name: str
    agents: int          # agents sharing each reused chunk (1 = single-request path)
    chunks: int          # reused chunks (shared blocks) per agent
    layers: int
    tokens: int          # n
    kv_heads: int
    head_dim: int
    rope_base: float
    r_num: int           # probe ratio r = r_num / r_den
    r_den: int
    check_layer: int
    heavy_frac: float
    heavy_kind: str      # "normal" | "student_t3"
    delta_kind: str      # "fixed" | "uniform" | "round"
    delta_fixed: int = 0
    delta_lo: int = 0
    delta_hi: int = 0
    seed: int = 0
    mu_std: float = 0.3
    xi_std: float = 0.05

    @property
    def b(self) -> int:
        """b = ceil(r n), in integers."""
        return -((-self.r_num * self.tokens) // self.r_den)

    @property
    def units(self) -> int:
        return self.agents * self.chunks

    def with_(self, **kw) -> "RepairConfig":
        return dataclasses.replace(self, **kw)


@dataclass(frozen=True)
class DiffConfig:
    name: str
    siblings: int
    layers: int
    tokens: int
    kv_heads: int
    head_dim: int
    block_tokens: int
    frac_lo: float
    frac_hi: float
    noise_std: float
    seed: int
    rope_base: float = 5e5
    page_tokens: int = 16

    @property
    def blocks(self) -> int:
        return self.tokens // self.block_tokens

    def with_(self, **kw) -> "DiffConfig":
        return dataclasses.replace(self, **kw)


@dataclass(frozen=True)
class LowRankConfig:
    name: str
    chunks: int
    layers: int
    tokens: int
    kv_heads: int
    q_heads: int
    head_dim: int
    rank: int
    draft_steps: int
    layer_begin: int
    budget_num: int      # repair budget rho = budget_num / budget_den of the rows
    budget_den: int
    a_std: float
    fresh_std: float
    seed: int

    @property
    def k_rows(self) -> int:
        """round(rho n), halves to even as Python's round does."""
        return int(round(self.budget_num * self.tokens / self.budget_den))

    def with_(self, **kw) -> "LowRankConfig":
        return dataclasses.replace(self, **kw)


@dataclass(frozen=True)
class AnchorConfig:
    name: str
    segments: int
    anchors: int
    layers: int
    tokens: int
    kv_heads: int
    head_dim: int
    rank: int
    rope_base: float
    tau: float           # reliability threshold
    noise_std: float     # source = the matching anchor's base state + N(0, noise_std^2)
    delta_std: float     # scale of the delta factor A_d
    seed: int

    def with_(self, **kw) -> "AnchorConfig":
        return dataclasses.replace(self, **kw)


REPAIR_TINY = RepairConfig("repair_tiny", agents=1, chunks=1, layers=2, tokens=256, kv_heads=4,
                           head_dim=64, rope_base=1e4, r_num=1, r_den=10, check_layer=1,
                           heavy_frac=0.05, heavy_kind="normal", delta_kind="fixed",
                           delta_fixed=137, seed=0)
REPAIR_LLAMA8B = RepairConfig("repair_llama8b", agents=1, chunks=1, layers=32, tokens=4096,
                              kv_heads=8, head_dim=128, rope_base=5e5, r_num=15, r_den=100,
                              check_layer=1, heavy_frac=0.03, heavy_kind="student_t3",
                              delta_kind="uniform", delta_lo=500, delta_hi=8000, seed=1)
ROUND_QWEN14B = RepairConfig("round_qwen14b", agents=8, chunks=8, layers=48, tokens=512,
                             kv_heads=8, head_dim=128, rope_base=1e6, r_num=1, r_den=10,
                             check_layer=1, heavy_frac=0.05, heavy_kind="normal",
                             delta_kind="round", delta_lo=200, delta_hi=3000, seed=2)
SIBLINGS_8B = DiffConfig("siblings_8b", siblings=16, layers=32, tokens=8192, kv_heads=8,
                         head_dim=128, block_tokens=16, frac_lo=0.03, frac_hi=0.09,
                         noise_std=0.2, seed=3)
LOWRANK_70B = LowRankConfig("lowrank_70b", chunks=4, layers=80, tokens=16384, kv_heads=8,
                            q_heads=64, head_dim=128, rank=16, draft_steps=2, layer_begin=1,
                            budget_num=5, budget_den=100, a_std=0.1, fresh_std=0.5, seed=4)

# Anchor-pool correction on Llama-3.1-8B-shaped caches: 2 shared segments of 4096 tokens,
# V = 10 anchors of rank 32 per layer and plane, tau = 0.32 (KVCMAS's GSM8K threshold).
ANCHOR_8B = AnchorConfig("anchor_8b", segments=2, anchors=10, layers=32, tokens=4096, kv_heads=8,
                         head_dim=128, rank=32, rope_base=5e5, tau=0.32, noise_std=0.3,
                         delta_std=0.1, seed=6)

CONFIGS = {c.name: c for c in (REPAIR_TINY, REPAIR_LLAMA8B, ROUND_QWEN14B, SIBLINGS_8B,
                               LOWRANK_70B)}


# ------------------------------------------------------------- generators

def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(stream)) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _normal(shape, std, g, device, dtype=torch.float32):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def repair_reuse(cfg: RepairConfig, device) -> dict:
    """Cached (reused) K and V ~ N(0,1) bf16, [chunks][L][n][H][D], and the per-unit
    position shift delta [agents*chunks] (unit index = agent*chunks + chunk)."""
    shape = (cfg.chunks, cfg.layers, cfg.tokens, cfg.kv_heads, cfg.head_dim)
    k = _normal(shape, 1.0, _gen(cfg.seed, 0, device), device, BF16)
    v = _normal(shape, 1.0, _gen(cfg.seed, 1, device), device, BF16)
    g = _gen(cfg.seed, 2, "cpu")
    if cfg.delta_kind == "fixed":
        delta = torch.full((cfg.units,), cfg.delta_fixed, dtype=torch.int32)
    elif cfg.delta_kind == "uniform":
        delta = torch.randint(cfg.delta_lo, cfg.delta_hi + 1, (cfg.units,), generator=g,
                              dtype=torch.int64).to(torch.int32)
    elif cfg.delta_kind == "round":
        # Each agent's prompt = private history H_a, then the shared blocks in a
        # per-agent order; shared block c sits at H_a + n * perm_a[c], and its cached
        # copy was encoded at canonical positions 0..n-1.
        hist = torch.randint(cfg.delta_lo, cfg.delta_hi + 1, (cfg.agents,), generator=g)
        rows = []
        for a in range(cfg.agents):
            perm = torch.randperm(cfg.chunks, generator=g)
            rows.append(hist[a] + cfg.tokens * perm)
        delta = torch.stack(rows).reshape(-1).to(torch.int32)
    else:
        raise ValueError(cfg.delta_kind)
    return {"k_reuse": k, "v_reuse": v, "delta": delta.to(device)}


def repair_residual(cfg: RepairConfig, unit: int, device) -> dict:
    """Residual draws of one (agent, chunk) unit: mu_k, mu_v [L][H][D] ~ N(0, mu_std^2);
    xi_k, xi_v [L][n][H][D] ~ N(0, xi_std^2) except on the unit's heavy tokens (the same
    tokens for K, V and every layer), which take the heavy-tailed draw instead."""
    g = _gen(cfg.seed, 100 + unit, device)
    L, n, H, D = cfg.layers, cfg.tokens, cfg.kv_heads, cfg.head_dim
    mu_k = _normal((L, H, D), cfg.mu_std, g, device)
    mu_v = _normal((L, H, D), cfg.mu_std, g, device)
    heavy_count = int(round(cfg.heavy_frac * n))
    heavy = torch.randperm(n, generator=g, device=device)[:heavy_count]
    out = {"mu_k": mu_k, "mu_v": mu_v, "heavy": heavy}
    for name in ("xi_k", "xi_v"):
        xi = _normal((L, n, H, D), cfg.xi_std, g, device)
        if heavy_count:
            if cfg.heavy_kind == "normal":
                hv = _normal((L, heavy_count, H, D), 1.0, g, device)
            elif cfg.heavy_kind == "student_t3":
                # t(3) = Z / sqrt(chi2_3 / 3), chi2_3 = sum of three squared normals.
                z = torch.randn((L, heavy_count, H, D), generator=g, device=device)
                c = torch.randn((3, L, heavy_count, H, D), generator=g, device=device)
                hv = z / torch.sqrt((c * c).sum(0) / 3.0)
            else:
                raise ValueError(cfg.heavy_kind)
            xi[:, heavy] = hv
        out[name] = xi
    return out


def diff_inputs(cfg: DiffConfig, device) -> dict:
    """Master K/V [L][n][H][D] ~ N(0,1) bf16 and siblings [S][L][n][H][D]: copies of the
    master in which a fraction f_s ~ U[frac_lo, frac_hi] of the token blocks (the same
    blocks in every layer, head and plane) is redrawn as bf16(master + N(0, std^2))."""
    L, n, H, D = cfg.layers, cfg.tokens, cfg.kv_heads, cfg.head_dim
    bt = cfg.block_tokens
    mk = _normal((L, n, H, D), 1.0, _gen(cfg.seed, 0, device), device, BF16)
    mv = _normal((L, n, H, D), 1.0, _gen(cfg.seed, 1, device), device, BF16)
    sk = mk.unsqueeze(0).repeat(cfg.siblings, 1, 1, 1, 1)
    sv = mv.unsqueeze(0).repeat(cfg.siblings, 1, 1, 1, 1)
    gsel = _gen(cfg.seed, 2, "cpu")
    dirty_blocks = []
    for s in range(cfg.siblings):
        f = cfg.frac_lo + (cfg.frac_hi - cfg.frac_lo) * torch.rand((), generator=gsel).item()
        m = max(1, int(round(f * cfg.blocks)))
        blocks = torch.randperm(cfg.blocks, generator=gsel)[:m].sort().values
        dirty_blocks.append(blocks)
        g = _gen(cfg.seed, 100 + s, device)
        for plane_s, plane_m in ((sk, mk), (sv, mv)):
            sel = plane_m.view(L, cfg.blocks, bt, H, D)[:, blocks.to(device)]
            noise = _normal(sel.shape, cfg.noise_std, g, device)
            plane_s[s].view(L, cfg.blocks, bt, H, D)[:, blocks.to(device)] = \
                (sel.float() + noise).to(BF16)
    return {"master_k": mk, "master_v": mv, "sib_k": sk, "sib_v": sv,
            "dirty_blocks": dirty_blocks}


def restore_inputs(cfg: DiffConfig, device, skip: float = 0.0, spare_pages: int = 0) -> dict:
    """Restore targets of the siblings: a shift delta[s] per sibling (sibling 0 keeps its
    positions, the others ~ U{1 .. 4n}) and a paged slot mapping [S][n]: the pool holds
    S*n/page + spare_pages pages of `page_tokens` rows, every (sibling, page) gets a
    distinct pool page drawn at random, token t sits at row t % page of its page.  A
    fraction `skip` of the tokens is left unmapped (slot -1)."""
    S, n, pg = cfg.siblings, cfg.tokens, cfg.page_tokens
    g = _gen(cfg.seed, 500, "cpu")
    delta = torch.randint(1, 4 * n + 1, (S,), generator=g, dtype=torch.int64)
    delta[0] = 0
    pages = S * ((n + pg - 1) // pg) + spare_pages
    perm = torch.randperm(pages, generator=g)[: S * ((n + pg - 1) // pg)].view(S, -1)
    t = torch.arange(n)
    slot = perm[:, t // pg] * pg + (t % pg)
    if skip > 0:
        slot[torch.rand((S, n), generator=g) < skip] = -1
    return {"delta": delta.to(torch.int32).to(device), "slot_mapping": slot.to(torch.int32).to(device),
            "slots": pages * pg}


def anchor_inputs(cfg: AnchorConfig, device) -> dict:
    """Draws per segment c and plane p: anchors' base factors a_c_p ~ N(0,1) [C][V][L][n][r]
    and b_ct_p ~ N(0, 1/r) [C][V][L][F][r] (base rows of unit variance); delta factors
    a_d_p ~ N(0, delta_std^2), b_dt_p ~ N(0, 1/r); noise_p ~ N(0, noise_std^2) [C][L][n][H][D]
    (bf16); the anchor each segment resembles, match[c] = c mod V (the source rows are
    composed from these draws by the caller: the base state of anchor match[c] plus the
    noise); key shifts delta ~ U{500..8000}."""
    C, V, L, n, r = cfg.segments, cfg.anchors, cfg.layers, cfg.tokens, cfg.rank
    F = cfg.kv_heads * cfg.head_dim
    out = {}
    bstd = 1.0 / float(r) ** 0.5
    for pi, p in enumerate(("k", "v")):
        base = 100 * (pi + 1)
        out[f"a_c_{p}"] = _normal((C, V, L, n, r), 1.0, _gen(cfg.seed, base + 1, device), device, BF16)
        out[f"b_ct_{p}"] = _normal((C, V, L, F, r), bstd, _gen(cfg.seed, base + 2, device), device, BF16)
        out[f"a_d_{p}"] = _normal((C, V, L, n, r), cfg.delta_std, _gen(cfg.seed, base + 3, device), device, BF16)
        out[f"b_dt_{p}"] = _normal((C, V, L, F, r), bstd, _gen(cfg.seed, base + 4, device), device, BF16)
        out[f"noise_{p}"] = _normal((C, L, n, cfg.kv_heads, cfg.head_dim), cfg.noise_std,
                                    _gen(cfg.seed, base + 5, device), device, BF16)
    out["match"] = [c % V for c in range(C)]
    gd = _gen(cfg.seed, 99, "cpu")
    out["delta"] = torch.randint(500, 8001, (C,), generator=gd, dtype=torch.int64).to(torch.int32).to(device)
    return out


def lowrank_inputs(cfg: LowRankConfig, device, planes=("k", "v")) -> dict:
    """x ~ N(0,1) [C][L][n][H][D]; A ~ N(0, a_std^2) [C][L][H][n][r]; B ~ N(0,1)
    [C][L][H][r][D] per plane; q ~ N(0,1) [C][L][T][Hq][D]; fresh = bf16(x + N(0, fresh_std^2))."""
    C, L, n, H, D, r = cfg.chunks, cfg.layers, cfg.tokens, cfg.kv_heads, cfg.head_dim, cfg.rank
    out = {}
    for pi, p in enumerate(planes):
        g = _gen(cfg.seed, 10 * pi, device)
        x = _normal((C, L, n, H, D), 1.0, g, device, BF16)
        out[f"x_{p}"] = x
        out[f"a_{p}"] = _normal((C, L, H, n, r), cfg.a_std, _gen(cfg.seed, 10 * pi + 1, device),
                                device, BF16)
        out[f"b_{p}"] = _normal((C, L, H, r, D), 1.0, _gen(cfg.seed, 10 * pi + 2, device),
                                device, BF16)
        gf = _gen(cfg.seed, 10 * pi + 3, device)
        fresh = torch.empty_like(x)
        for c in range(C):  # chunk by chunk to bound the float32 temporary
            fresh[c] = (x[c].float() + _normal(x[c].shape, cfg.fresh_std, gf, device)).to(BF16)
        out[f"fresh_{p}"] = fresh
    out["q"] = _normal((C, L, cfg.draft_steps, cfg.q_heads, D), 1.0, _gen(cfg.seed, 99, device),
                       device, BF16)
    return out


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (copied to host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def from_bits(a, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(BF16).to(device)
