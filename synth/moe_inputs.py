"""Seeded synthetic inputs: checkpoint-layout expert weights, hidden states and router outputs.

Shapes and value ranges follow the five workloads of the routed-MoE pages
(sglang ``moe_b12x_next.py`` adapter: DSV4 E=384, H=7168, per-rank I=576,
top-6, MXFP4 weights; vLLM ``hybrid_loader.py``: GLM-5.2 E=256, H=6144, I=512,
top-8, NVFP4 + NF3).  Nothing here decodes or computes: codes and scales are
uniform random bytes in the checkpoint tensor layouts the pages list
(``_convert_layer`` shape checks; ``HybridNvFp4MoE.create_weights``, whose "v3" kept tier is
MXFP4 for hybrid-mapped layers).

Checkpoint layouts (row-major, contiguous):
  MXFP4: w13 [E, 2I, H/2] u8 (two E2M1 per byte), s13 [E, 2I, H/32] u8 (E8M0),
         w2  [E, H, I/2]  u8,                     s2  [E, H, I/32]  u8.
  NVFP4: w13 [E, 2I, H/2], s13 [E, 2I, H/16] u8 (E4M3), g13 [E] f32,
         w2  [E, H, I/2],  s2  [E, H, I/16] u8 (E4M3),  g2  [E] f32.
  NF3:   w13 [E, 2I, 3H/8] u8 (8 codes per 3 bytes), s13 [E, 2I, H/32] u8 (E4M3),
         w2  [E, H, 3I/8],                          s2  [E, H, I/32] u8 (E4M3).
The w13 rows are [up; gate] (``W13Layout.W13``, the adapter's
``load_up_proj_weight_first`` stacking) unless ``layout`` says gate first.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

W13_UP_GATE = 0
W13_GATE_UP = 1

TIER_NVFP4 = 4
TIER_NF3 = 3


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    E: int
    H: int
    I: int
    topk: int
    quant: str                 # "w4a8_mxfp4" | "w4a16_nvfp4" | "w4a8_nvfp4" | "w4a4_nvfp4" |
                               # "hybrid" | "hybrid_mx"
    swiglu_limit: float        # +inf = no clamp
    m_list: tuple
    routing: str = "uniform"   # "uniform" | "zipf"
    zipf_s: float = 0.0
    weight_rule: str = "sigmoid_norm"   # "softmax" | "sigmoid_norm"
    weight_mult: float = 1.0
    pad_frac: float = 0.0      # last floor(M * pad_frac) rows are padding (id -1)
    scale_lo: int = 0          # scale byte range (E8M0 bytes or E4M3 codes)
    scale_hi: int = 0
    n_nvfp4: int = 0           # hybrid: experts in the kept (NVFP4 or MXFP4) tier
    kept_scale_lo: int = 0     # hybrid_mx: E8M0 byte range of the MXFP4 kept tier
    kept_scale_hi: int = 0
    ep_local: int = 0          # >0: ids drawn over ep_global experts and masked to the local ones
    ep_global: int = 0
    seed_base: int = 0


INF = float("inf")

CONFIGS = {
    # Tiny W4A8: E8 H256 I128 top-2, M=4, E8M0 exponents 2^-4..2^0, softmax weights, seed 0.
    "tiny_w4a8": MoEConfig("tiny_w4a8", E=8, H=256, I=128, topk=2, quant="w4a8_mxfp4",
                           swiglu_limit=7.0, m_list=(4,), weight_rule="softmax",
                           scale_lo=123, scale_hi=127, seed_base=0),
    # Decode / verify slice: E384 H7168 I576 top-6, E8M0 2^-8..2^-2, 2.5x renormalised sigmoid
    # weights, last 25 % rows padding.
    "decode_w4a8": MoEConfig("decode_w4a8", E=384, H=7168, I=576, topk=6, quant="w4a8_mxfp4",
                             swiglu_limit=7.0, m_list=(1, 2, 3, 4, 5, 6, 7, 8, 10, 12, 14, 16),
                             weight_rule="sigmoid_norm", weight_mult=2.5, pad_frac=0.25,
                             scale_lo=119, scale_hi=125, seed_base=2000),
    # Prefill ladder, same format; uniform routing.
    "prefill_w4a8": MoEConfig("prefill_w4a8", E=384, H=7168, I=576, topk=6, quant="w4a8_mxfp4",
                              swiglu_limit=7.0, m_list=(128, 256, 512, 1024, 2048, 4096),
                              weight_rule="sigmoid_norm", weight_mult=2.5,
                              scale_lo=119, scale_hi=125, seed_base=3000),
    # Prefill ladder with Zipf(s=1.0) load imbalance.
    "prefill_w4a8_zipf": MoEConfig("prefill_w4a8_zipf", E=384, H=7168, I=576, topk=6,
                                   quant="w4a8_mxfp4", swiglu_limit=7.0,
                                   m_list=(128, 256, 512, 1024, 2048, 4096), routing="zipf",
                                   zipf_s=1.0, weight_rule="sigmoid_norm", weight_mult=2.5,
                                   scale_lo=119, scale_hi=125, seed_base=3001),
    # EP2 slice: 192 locally owned experts at I=1152; foreign ids masked to weight 0.
    "prefill_w4a8_ep_i1152": MoEConfig("prefill_w4a8_ep_i1152", E=192, H=7168, I=1152, topk=6,
                                       quant="w4a8_mxfp4", swiglu_limit=7.0,
                                       m_list=(128, 256, 512, 1024, 2048, 4096),
                                       weight_rule="sigmoid_norm", weight_mult=2.5,
                                       scale_lo=119, scale_hi=125, ep_local=192, ep_global=384,
                                       seed_base=3002),
    # NVFP4 W4A16: E256 H6144 I512 top-8; E4M3 block scales 2^-6..2^2, g ~ U(0.5,2)/448.
    "w4a16_nvfp4": MoEConfig("w4a16_nvfp4", E=256, H=6144, I=512, topk=8, quant="w4a16_nvfp4",
                             swiglu_limit=INF, m_list=(1, 8, 64, 512, 2048, 8192),
                             weight_rule="sigmoid_norm", scale_lo=0x08, scale_hi=0x48,
                             seed_base=4000),
    # Hybrid: 64 NVFP4 + 192 NF3 experts, Zipf(s=0.8) routing, deterministic combine.
    "hybrid_nvfp4_nf3": MoEConfig("hybrid_nvfp4_nf3", E=256, H=6144, I=512, topk=8,
                                  quant="hybrid", swiglu_limit=INF, m_list=(8, 2048),
                                  routing="zipf", zipf_s=0.8, weight_rule="sigmoid_norm",
                                  scale_lo=0x08, scale_hi=0x48, n_nvfp4=64, seed_base=5000),
    # NVFP4 weights with MXFP8 activations (B12xExperts "w4a8_nvfp4"): the NVFP4 layer above
    # with per-expert activation global scales.
    "w4a8_nvfp4": MoEConfig("w4a8_nvfp4", E=256, H=6144, I=512, topk=8, quant="w4a8_nvfp4",
                            swiglu_limit=INF, m_list=(1, 8, 64, 512, 2048),
                            weight_rule="sigmoid_norm", scale_lo=0x08, scale_hi=0x48,
                            seed_base=4100),
    # NVFP4 weights with NVFP4 activations (B12xExperts "nvfp4", W4A4): the same layer and
    # activation global scales.
    "w4a4_nvfp4": MoEConfig("w4a4_nvfp4", E=256, H=6144, I=512, topk=8, quant="w4a4_nvfp4",
                            swiglu_limit=INF, m_list=(1, 8, 64, 512, 2048),
                            weight_rule="sigmoid_norm", scale_lo=0x08, scale_hi=0x48,
                            seed_base=4200),
    # Hybrid "v3": the same layer with the 64 kept experts in MXFP4 (E8M0 2^-8..2^-2) and bf16
    # activations; NF3 tier as above.
    "hybrid_mxfp4_nf3": MoEConfig("hybrid_mxfp4_nf3", E=256, H=6144, I=512, topk=8,
                                  quant="hybrid_mx", swiglu_limit=INF, m_list=(8, 2048),
                                  routing="zipf", zipf_s=0.8, weight_rule="sigmoid_norm",
                                  scale_lo=0x08, scale_hi=0x48, n_nvfp4=64, kept_scale_lo=119,
                                  kept_scale_hi=125, seed_base=5100),
}


@dataclasses.dataclass
class Checkpoint:
    """Checkpoint-layout tensors of one MoE layer (numpy, host)."""
    quant: str                      # "mxfp4" | "nvfp4" | "w4a8_nvfp4" | "w4a4_nvfp4" | "nf3" |
                                    # "hybrid"
    E: int
    H: int
    I: int
    layout: int = W13_UP_GATE
    w13: Optional[np.ndarray] = None
    s13: Optional[np.ndarray] = None
    w2: Optional[np.ndarray] = None
    s2: Optional[np.ndarray] = None
    g13: Optional[np.ndarray] = None
    g2: Optional[np.ndarray] = None
    # w4a8_nvfp4 only: per-expert activation global scales of fc1's / fc2's input (fp32 [E])
    a13: Optional[np.ndarray] = None
    a2: Optional[np.ndarray] = None
    # hybrid only
    tier: Optional[np.ndarray] = None        # [E] int8, TIER_NVFP4 or TIER_NF3
    nv: Optional["Checkpoint"] = None        # kept tier (NVFP4, or MXFP4), compact over its experts
    nf: Optional["Checkpoint"] = None        # NF3 tier, compact over its experts
    # hybrid with an MXFP4 kept tier: the layer's static FP8 input scales (fp32 scalars)
    in13: Optional[float] = None
    in2: Optional[float] = None


def _bytes(rng, shape, lo=0, hi=255):
    return rng.integers(lo, hi + 1, size=shape, dtype=np.uint8)


def make_fp4_checkpoint(rng, kind, E, H, I, scale_lo, scale_hi, layout=W13_UP_GATE):
    """Random E2M1 codes (every nibble uniform over 16 codes) and random scale bytes.

    kind "mxfp4": E8M0 scale bytes per 32 uniform in [scale_lo, scale_hi].
    kind "nvfp4": E4M3 scale codes per 16 uniform in [scale_lo, scale_hi] plus one fp32 global
    scale per expert and matrix, U(0.5, 2)/448.
    """
    blk = 32 if kind == "mxfp4" else 16
    ck = Checkpoint(quant=kind, E=E, H=H, I=I, layout=layout)
    ck.w13 = _bytes(rng, (E, 2 * I, H // 2))
    ck.s13 = _bytes(rng, (E, 2 * I, H // blk), scale_lo, scale_hi)
    ck.w2 = _bytes(rng, (E, H, I // 2))
    ck.s2 = _bytes(rng, (E, H, I // blk), scale_lo, scale_hi)
    if kind == "nvfp4":
        ck.g13 = (rng.uniform(0.5, 2.0, size=E) / 448.0).astype(np.float32)
        ck.g2 = (rng.uniform(0.5, 2.0, size=E) / 448.0).astype(np.float32)
    return ck


def make_nf3_checkpoint(rng, E, H, I, scale_lo, scale_hi, layout=W13_UP_GATE):
    """NF3 codes uniform over the 8 LUT entries (uniform random packed bytes make every 3-bit
    field uniform and independent) and E4M3 scale codes per group of 32 along K."""
    ck = Checkpoint(quant="nf3", E=E, H=H, I=I, layout=layout)
    ck.w13 = _bytes(rng, (E, 2 * I, H // 8 * 3))
    ck.s13 = _bytes(rng, (E, 2 * I, H // 32), scale_lo, scale_hi)
    ck.w2 = _bytes(rng, (E, H, I // 8 * 3))
    ck.s2 = _bytes(rng, (E, H, I // 32), scale_lo, scale_hi)
    return ck


def make_checkpoint(cfg: MoEConfig, seed: Optional[int] = None, E: Optional[int] = None,
                    H: Optional[int] = None, I: Optional[int] = None,
                    layout: int = W13_UP_GATE) -> Checkpoint:
    """Weights of one layer of ``cfg`` (shape overrides allow small cases of the same recipe)."""
    E = cfg.E if E is None else E
    H = cfg.H if H is None else H
    I = cfg.I if I is None else I
    rng = np.random.default_rng(cfg.seed_base if seed is None else seed)
    if cfg.quant == "w4a8_mxfp4":
        return make_fp4_checkpoint(rng, "mxfp4", E, H, I, cfg.scale_lo, cfg.scale_hi, layout)
    if cfg.quant == "w4a16_nvfp4":
        return make_fp4_checkpoint(rng, "nvfp4", E, H, I, cfg.scale_lo, cfg.scale_hi, layout)
    if cfg.quant in ("w4a8_nvfp4", "w4a4_nvfp4"):
        # NVFP4 weights with MXFP8 activations: activation global scales 1 / input_scale =
        # 6 x 448 / calibration amax, drawn log-uniformly over a factor 4 around an amax of 5
        # for x (N(0,1) rows) and 8 for h (the full-size layer's SwiGLU outputs reach ~6)
        ck = make_fp4_checkpoint(rng, "nvfp4", E, H, I, cfg.scale_lo, cfg.scale_hi, layout)
        ck.quant = cfg.quant
        ck.a13 = (2688.0 / 5.0 * 2.0 ** rng.uniform(-1, 1, size=E)).astype(np.float32)
        ck.a2 = (2688.0 / 8.0 * 2.0 ** rng.uniform(-1, 1, size=E)).astype(np.float32)
        return ck
    if cfg.quant in ("hybrid", "hybrid_mx"):
        n4 = min(cfg.n_nvfp4, E) if E != cfg.E else cfg.n_nvfp4
        # Which experts are kept in NVFP4 is a seeded random subset (the pages keep the top-64
        # by an importance score that synthetic weights do not have).
        kept = np.sort(rng.permutation(E)[:n4])
        tier = np.full(E, TIER_NF3, dtype=np.int8)
        tier[kept] = TIER_NVFP4
        ck = Checkpoint(quant="hybrid", E=E, H=H, I=I, layout=layout, tier=tier)
        if cfg.quant == "hybrid_mx":
            ck.nv = make_fp4_checkpoint(rng, "mxfp4", n4, H, I, cfg.kept_scale_lo,
                                        cfg.kept_scale_hi, layout)
        else:
            ck.nv = make_fp4_checkpoint(rng, "nvfp4", n4, H, I, cfg.scale_lo, cfg.scale_hi,
                                        layout)
        ck.nf = make_nf3_checkpoint(rng, E - n4, H, I, cfg.scale_lo, cfg.scale_hi, layout)
        if cfg.quant == "hybrid_mx":
            # w13_input_scale / w2_input_scale of the kept tier's A8 opt-in: calibration amax
            # / 448, log-uniform over a factor 2 around an amax of 5 for x and 8 for h
            ck.in13 = float(np.float32(5.0 / 448.0 * 2.0 ** rng.uniform(-0.5, 0.5)))
            ck.in2 = float(np.float32(8.0 / 448.0 * 2.0 ** rng.uniform(-0.5, 0.5)))
        return ck
    raise ValueError(cfg.quant)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def make_x(rng, M: int, H: int) -> np.ndarray:
    """Hidden states, bf16 ~ N(0,1), returned as uint16 bit patterns [M, H]."""
    return f32_to_bf16_bits(rng.standard_normal((M, H), dtype=np.float32))


def uniform_topk(rng, M: int, E: int, k: int) -> np.ndarray:
    """k distinct experts per row, uniform without replacement (argsort of uniform keys)."""
    return np.argsort(rng.random((M, E)), axis=1)[:, :k].astype(np.int32)


def zipf_topk(rng, M: int, E: int, k: int, s: float) -> np.ndarray:
    """k distinct experts per row with P(rank r) ~ r^-s, drawn without replacement.

    Gumbel-top-k over log-probabilities -s*log(r) (equivalent to sequential sampling without
    replacement); ranks are mapped to expert ids by a seeded permutation so the hot experts are
    spread over the id range.
    """
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    g = rng.gumbel(size=(M, E))
    ranks = np.argsort(-(logp[None, :] + g), axis=1)[:, :k]
    rank_to_id = rng.permutation(E).astype(np.int32)
    return rank_to_id[ranks]


def router_weights(rng, M: int, k: int, rule: str, mult: float) -> np.ndarray:
    z = rng.standard_normal((M, k))
    if rule == "softmax":
        p = np.exp(z - z.max(axis=1, keepdims=True))
        w = p / p.sum(axis=1, keepdims=True)
    elif rule == "sigmoid_norm":
        sg = 1.0 / (1.0 + np.exp(-z))
        w = sg / sg.sum(axis=1, keepdims=True)
    else:
        raise ValueError(rule)
    return (w * mult).astype(np.float32)


def ep_mask_foreign(ids_global: np.ndarray, w: np.ndarray, offset: int, num_local: int):
    """Router output of the whole model -> router output one expert-parallel rank sees.

    The rank owns the global experts [offset, offset + num_local).  An owned slot keeps its
    weight and becomes local id (global - offset).  Every other slot - another rank's expert or
    a padding id - gets weight 0 and a stand-in local id: the smallest owned local id in its
    own row; if the row owns none, the smallest owned local id anywhere in the batch; if the
    batch owns none, 0.  (The EP adapter's remap rule, moe_b12x_next.py ``ep_remap``.)"""
    gid = np.asarray(ids_global, dtype=np.int64)
    local = gid - offset
    owned = (local >= 0) & (local < num_local)
    batch_lowest = int(local[owned].min()) if owned.any() else 0
    ids = np.empty(gid.shape, dtype=np.int32)
    for t in range(gid.shape[0]):
        mine = local[t][owned[t]]
        stand_in = int(mine.min()) if mine.size else batch_lowest
        ids[t] = np.where(owned[t], local[t], stand_in)
    return ids, np.where(owned, np.asarray(w, dtype=np.float32), np.float32(0)).astype(np.float32)


def make_routing(cfg: MoEConfig, M: int, seed: Optional[int] = None, E: Optional[int] = None):
    """Router outputs (topk_ids int32 [M,k], topk_weights fp32 [M,k]) for ``cfg`` at ``M`` rows."""
    rng = np.random.default_rng(cfg.seed_base + M if seed is None else seed)
    k = cfg.topk
    E = cfg.E if E is None else E
    if cfg.ep_local:
        ids_g = uniform_topk(rng, M, cfg.ep_global, k)
        w = router_weights(rng, M, k, cfg.weight_rule, cfg.weight_mult)
        return ep_mask_foreign(ids_g, w, 0, cfg.ep_local)
    if cfg.routing == "zipf":
        ids = zipf_topk(rng, M, E, k, cfg.zipf_s)
    else:
        ids = uniform_topk(rng, M, E, k)
    w = router_weights(rng, M, k, cfg.weight_rule, cfg.weight_mult)
    n_pad = int(M * cfg.pad_frac)
    if n_pad:
        ids[M - n_pad:, :] = -1          # CUDA-graph padding rows; their weights stay nonzero
    return ids, w


def make_inputs(cfg: MoEConfig, M: int, seed: Optional[int] = None, H: Optional[int] = None,
                E: Optional[int] = None):
    """x (bf16 bits [M,H]), topk_ids, topk_weights for one call."""
    H = cfg.H if H is None else H
    rng = np.random.default_rng((cfg.seed_base + M if seed is None else seed) + 7919)
    x = make_x(rng, M, H)
    ids, w = make_routing(cfg, M, seed=seed, E=E)
    return x, ids, w
