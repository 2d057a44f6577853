"""The routed-MoE forward by definition, in fp64 on the CPU (test infrastructure only).

out[t] = sum_j w[t,j] * expert_{id[t,j]}(x[t]),  expert(x) = W2 . act(gate(x), up(x))

with gate/up the two halves of fc1 = W13 . x (hybrid_loader.py ``_apply_ref``; vLLM B12xExperts
``apply``).  Ids outside [0, E), the -1 of CUDA-graph padding rows included, contribute nothing
(moe_b12x_next.py, knob ``_DIRECT_IDS``: the kernels skip ids outside [0, E) and padding rows
come out 0).

Readings where the pages are silent (each one is listed with its reason in the design notes):
  * SwiGLU clamp: gate' = min(gate, L), up' = clamp(up, -L, L),
    h = gate' * sigmoid(alpha * gate') * (up' + beta), alpha = 1 and beta = 0 unless given;
    L = +inf means no clamp, which is the plain silu(g) * u of ``_apply_ref``.
  * W4A8: x is quantised to MXFP8 before fc1, h is quantised to MXFP8 before fc2 (from the
    unrounded SwiGLU output).  W4A16: x enters as bf16, h is rounded to bf16 before fc2.
  * NVFP4 weights with MXFP8 or NVFP4 activations: the activations (x and h) are multiplied by
    the expert's activation global scale in fp32, quantised (OCP MX rule, or NVFP4 blocks of 16
    with an E4M3 scale of vmax / 6), dequantised and divided by the scale.
  * Hybrid layers: the kept tier is NVFP4, or MXFP4 for hybrid_loader.py's "v3" kept format
    (``_build_kept_mxfp4``, A16 default); either way with bf16 activations, except for the A8
    opt-in of the MXFP4 kept tier (``kept_a8``): its experts' x and h are static per-tensor FP8
    with the layer's two input scales (codecs.fp8_static_quantize), h taken from the unrounded
    SwiGLU output as for W4A8; the NF3 experts keep bf16 activations.
  * The result is accumulated in fp64 over the top-k slots and rounded to bf16 once.
  * Routing order: the slots of expert e are listed in ascending (t, j) order (stable
    counting sort).
"""
from __future__ import annotations

import math

import numpy as np

from . import codecs as C

W13_UP_GATE = 0
W13_GATE_UP = 1
TIER_NVFP4 = 4
TIER_NF3 = 3


# ---------------------------------------------------------------------------- routing

def route(topk_ids: np.ndarray, E: int):
    """Routing by definition.

    Valid slots are the flat indices f = t*k + j with 0 <= id < E.
      cnt[e]     number of valid slots with id e
      off[e]     exclusive prefix sum of cnt (off[E] = S, the number of valid slots)
      perm[p]    flat slot index at position p; the slots of expert e occupy
                 off[e] .. off[e+1]-1 in ascending flat order
      slot_of[f] position of flat slot f in perm, -1 for dropped ids
    Pinned by tests/test_oracle_moe.py (hand-worked case in tests/golden/routing.txt and a
    pure-Python brute force).
    """
    flat = np.asarray(topk_ids, dtype=np.int64).ravel()
    valid = (flat >= 0) & (flat < E)
    cnt = np.bincount(flat[valid], minlength=E).astype(np.int32)
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(cnt)
    key = np.where(valid, flat, E)
    order = np.argsort(key, kind="stable")
    S = int(valid.sum())
    perm = order[:S].astype(np.int32)
    slot_of = np.full(flat.shape[0], -1, dtype=np.int32)
    slot_of[perm] = np.arange(S, dtype=np.int32)
    return cnt, off, perm, slot_of


# ---------------------------------------------------------------------------- activation

def swiglu(gate, up, limit=math.inf, alpha=1.0, beta=0.0):
    """Clamped SwiGLU (reading above).  Pinned by closed forms in tests/test_oracle_moe.py."""
    g = np.minimum(np.asarray(gate, dtype=np.float64), limit)
    u = np.clip(np.asarray(up, dtype=np.float64), -limit, limit)
    with np.errstate(over="ignore"):      # exp overflow for a very negative gate: sigmoid 0
        return g * (1.0 / (1.0 + np.exp(-alpha * g))) * (u + beta)


# ---------------------------------------------------------------------------- weights

def _fp4_values(packed: np.ndarray) -> np.ndarray:
    return C.E2M1_TABLE[C.unpack_fp4(packed)]


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[R, K/2] E2M1 bytes, [R, K/32] E8M0 bytes -> [R, K] fp64: E2M1(code) * 2^(s-127)."""
    v = _fp4_values(packed)
    return v * np.repeat(C.e8m0_value(scales), 32, axis=1)


def dequant_nvfp4(packed: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    """[R, K/2] E2M1 bytes, [R, K/16] E4M3 bytes, fp32 global -> E2M1 * E4M3(s) * g.
    Reading: the per-expert ``weight_scale_2`` multiplies (one global per matrix)."""
    v = _fp4_values(packed)
    return v * np.repeat(C.e4m3_decode(scales), 16, axis=1) * float(g)


def dequant_nf3(packed: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    return C.nf3_dequant(packed, scales, K)


def tier_local_index(tier: np.ndarray):
    """Hybrid layer: expert e -> (tier, index among the experts of that tier in ascending e),
    the compact two-group storage of hybrid_loader.py (``remap``)."""
    out = {}
    n = {TIER_NVFP4: 0, TIER_NF3: 0}
    for e, t in enumerate(np.asarray(tier).tolist()):
        out[e] = (int(t), n[int(t)])
        n[int(t)] += 1
    return out


def expert_weights(ck, e: int):
    """Dequantised (W13 [2I, H], W2 [H, I], kind) of expert e of a synth Checkpoint."""
    H, I = ck.H, ck.I
    if ck.quant == "mxfp4":
        return dequant_mxfp4(ck.w13[e], ck.s13[e]), dequant_mxfp4(ck.w2[e], ck.s2[e]), "mxfp4"
    if ck.quant in ("nvfp4", "w4a8_nvfp4", "w4a4_nvfp4"):
        return (dequant_nvfp4(ck.w13[e], ck.s13[e], ck.g13[e]),
                dequant_nvfp4(ck.w2[e], ck.s2[e], ck.g2[e]), "nvfp4")
    if ck.quant == "nf3":
        return dequant_nf3(ck.w13[e], ck.s13[e], H), dequant_nf3(ck.w2[e], ck.s2[e], I), "nf3"
    if ck.quant == "hybrid":
        t, li = tier_local_index(ck.tier)[e]
        sub = ck.nv if t == TIER_NVFP4 else ck.nf
        return expert_weights(sub, li)
    raise ValueError(ck.quant)


def split_w13(g13: np.ndarray, I: int, layout: int):
    """fc1 output [.., 2I] -> (gate, up) according to the stacking order of W13."""
    first, second = g13[..., :I], g13[..., I:]
    return (second, first) if layout == W13_UP_GATE else (first, second)


# ---------------------------------------------------------------------------- forward

def activation_a8(ck) -> bool:
    """MXFP8 activations: W4A8 (MXFP4 weights) and NVFP4 weights in the "w4a8_nvfp4" mode."""
    return ck.quant in ("mxfp4", "w4a8_nvfp4")


def act_gscale(ck, which: str):
    """Per-expert activation global scales [E] of fc1's ("a1") or fc2's ("a2") input, or None
    (B12xExperts ``_prepare_experts``: the NVFP4 modes with quantised activations take
    a1_gscale / a2_gscale)."""
    if ck.quant not in ("w4a8_nvfp4", "w4a4_nvfp4"):
        return None
    return ck.a13 if which == "a1" else ck.a2


def activation_nv4(ck) -> bool:
    """NVFP4 activations (W4A4: B12xExperts quant mode "nvfp4", kNvfp4Static weights with
    kNvfp4Dynamic activations)."""
    return ck.quant == "w4a4_nvfp4"


def nvfp4_act(v, a):
    """NVFP4 activations with the expert's global scale a: the fp32 product a * v quantised by
    codecs.nvfp4_quantize, dequantised and divided by a (reading: as for MXFP8 activations)."""
    a32 = np.float32(a)
    va = (a32 * np.asarray(v, dtype=np.float64).astype(np.float32)).astype(np.float32)
    q, s = C.nvfp4_quantize(va)
    return C.nvfp4_dequantize(q, s) / np.float64(a32)


def quantize_x(x_bits: np.ndarray, a8: bool, a=None):
    """x as the fc1 kernel sees it: MXFP8 (codes, scales, dequantised values) or bf16 values.
    With an activation global scale ``a`` (reading: it multiplies x in fp32 before the MX
    quantisation and divides the dequantised value) the values are MXFP8(fp32(a * x)) / a."""
    x = C.bf16_bits_to_f64(x_bits)
    if a8:
        if a is not None:
            xa = (np.float32(a) * x.astype(np.float32)).astype(np.float64)
            q, s = C.mxfp8_quantize(xa)
            return q, s, C.mxfp8_dequantize(q, s) / np.float64(np.float32(a))
        q, s = C.mxfp8_quantize(x)
        return q, s, C.mxfp8_dequantize(q, s)
    return None, None, x


def requant_h(h: np.ndarray, a8: bool, a=None) -> np.ndarray:
    """fc2's input: MXFP8 of h (of a * h, divided by a, with an activation global scale), or
    bf16(h) for 16-bit activations."""
    if a8:
        a64 = 1.0 if a is None else np.float64(np.float32(a))
        q, s = C.mxfp8_quantize(h * a64)
        return C.mxfp8_dequantize(q, s) / a64
    return C.bf16_round(h)


def kept_a8_scales(ck, e: int, kept_a8: bool):
    """(w13 input scale, w2 input scale) of expert e when the A8 opt-in of the MXFP4 kept tier
    applies to it (hybrid_loader.py ``_build_kept_mxfp4``, ``HYBRID_MX_A8``), else None."""
    if not kept_a8:
        return None
    assert ck.quant == "hybrid" and ck.nv.quant == "mxfp4", "A8 opt-in: MXFP4 kept tier only"
    t, _ = tier_local_index(ck.tier)[e]
    return (ck.in13, ck.in2) if t == TIER_NVFP4 else None


def slot_input(xin, w_slot, weight_on_input):
    """fc1 input and combine weight of slots: x and w, or with the router weight applied to the
    input (B12xExperts ``apply_router_weight_on_input``, W4A16 only) bf16(x * bf16(w)) and 1 -
    reading: the weight is cast to the activations' dtype and multiplies them in it."""
    if not weight_on_input:
        return xin, w_slot
    return C.bf16_round(xin * C.bf16_round(w_slot)[:, None]), np.ones_like(w_slot)


def moe_forward(ck, x_bits, topk_ids, topk_w, limit=math.inf, alpha=1.0, beta=0.0,
                rows=None, return_f64=False, weight_on_input=False, kept_a8=False):
    """Per-expert dgemm form.  ``rows`` restricts the output to a subset of token rows
    (the other rows are not computed and come back as NaN).  Returns bf16 bit patterns
    [M, H] (and the unrounded fp64 sum when ``return_f64``).  ``weight_on_input``: the router
    weights scale fc1's input instead of the expert outputs (16-bit activations only).
    Pinned by tests/test_oracle_moe.py against the brute-force loop, closed forms and the
    invariants (linearity in the weights, padding rows, token-order invariance, w13 halves)."""
    x_bits = np.asarray(x_bits)
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    M, k = ids.shape
    E, H, I = ck.E, ck.H, ck.I
    a8 = activation_a8(ck)
    assert not ((a8 or activation_nv4(ck) or kept_a8) and weight_on_input), \
        "router weights on the input need 16-bit activations"
    out = np.zeros((M, H), dtype=np.float64)
    row_mask = np.ones(M, dtype=bool)
    if rows is not None:
        row_mask[:] = False
        row_mask[np.asarray(rows)] = True
    a1, a2 = act_gscale(ck, "a1"), act_gscale(ck, "a2")
    nv4 = activation_nv4(ck)
    _, _, xhat = quantize_x(x_bits[row_mask] if rows is not None else x_bits, a8 and a1 is None)
    if rows is not None:
        full = np.full((M, H), np.nan)
        full[row_mask] = xhat
        xhat = full
    valid = (ids >= 0) & (ids < E) & row_mask[:, None]
    for e in np.unique(ids[valid]):
        sel = valid & (ids == e)
        t_idx, j_idx = np.nonzero(sel)
        W13, W2, _ = expert_weights(ck, int(e))
        xin, cw = slot_input(xhat[t_idx], w[t_idx, j_idx], weight_on_input)
        if nv4:                # NVFP4 activations with the expert's global scale
            xin = nvfp4_act(C.bf16_bits_to_f64(x_bits[t_idx]), a1[e])
        elif a1 is not None:   # MXFP8 activations with the expert's global scale
            xin = quantize_x(x_bits[t_idx], True, a1[e])[2]
        s8 = kept_a8_scales(ck, int(e), kept_a8)
        if s8 is not None:     # static per-tensor FP8 activations of the kept tier
            xin = C.fp8_static_quantize(C.bf16_bits_to_f64(x_bits[t_idx]), s8[0])[1]
        G = xin @ W13.T
        gate, up = split_w13(G, I, ck.layout)
        h = swiglu(gate, up, limit, alpha, beta)
        if s8 is not None:
            hh = C.fp8_static_quantize(h, s8[1])[1]
        else:
            hh = nvfp4_act(h, a2[e]) if nv4 else requant_h(h, a8, None if a2 is None else a2[e])
        y = hh @ W2.T
        np.add.at(out, t_idx, cw[:, None] * y)
    out[~row_mask] = np.nan
    bits = C.f64_to_bf16_bits(np.where(row_mask[:, None], out, 0.0))
    if return_f64:
        return bits, out
    return bits


def slot_intermediate(ck, x_bits, topk_ids, limit=math.inf, alpha=1.0, beta=0.0, topk_w=None,
                      weight_on_input=False, kept_a8=False):
    """The SwiGLU output h (fp64, before the fc2 quantisation) of every valid slot, in routing
    order (row p belongs to flat slot perm[p]); shape [S, I].  With ``weight_on_input`` the
    slots' inputs are scaled by ``topk_w`` as in moe_forward."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    M, k = ids.shape
    a8 = activation_a8(ck)
    a1 = act_gscale(ck, "a1")
    _, _, xhat = quantize_x(np.asarray(x_bits), a8 and a1 is None)
    _, off, perm, _ = route(ids, ck.E)
    out = np.zeros((perm.shape[0], ck.I))
    for e in range(ck.E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        W13, _, _ = expert_weights(ck, e)
        fl = perm[lo:hi]
        xin = xhat[fl // k]
        if activation_nv4(ck):
            xin = nvfp4_act(C.bf16_bits_to_f64(np.asarray(x_bits)[fl // k]), a1[e])
        elif a1 is not None:
            xin = quantize_x(np.asarray(x_bits)[fl // k], True, a1[e])[2]
        s8 = kept_a8_scales(ck, e, kept_a8)
        if s8 is not None:
            xin = C.fp8_static_quantize(C.bf16_bits_to_f64(np.asarray(x_bits)[fl // k]), s8[0])[1]
        if weight_on_input:
            xin, _ = slot_input(xin, np.asarray(topk_w, np.float64).reshape(-1)[fl], True)
        G = xin @ W13.T
        gate, up = split_w13(G, ck.I, ck.layout)
        out[lo:hi] = swiglu(gate, up, limit, alpha, beta)
    return out


def requant_alternatives(ck, x_bits, topk_ids, topk_w, limit=math.inf, alpha=1.0, beta=0.0,
                         rel=1e-4, rows=None, weight_on_input=False, kept_a8=False):
    """Legitimate alternatives of the fc2 operand's rounding (reading: where floating point
    decides a quantised code, arithmetic exact to a relative error `rel` may land on either
    neighbour of a near-midpoint value).  For every output row (or the given rows) returns a list
    of fp64 vectors d, one per ambiguous intermediate element of that row's slots, such that
    rounding that element the other way changes the row's unrounded output by exactly d."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    M, k = ids.shape
    a8 = activation_a8(ck)
    h = slot_intermediate(ck, x_bits, ids, limit, alpha, beta, topk_w, weight_on_input, kept_a8)
    _, _, perm, _ = route(ids, ck.E)
    a2 = act_gscale(ck, "a2")
    if activation_nv4(ck):
        sc = np.float32(a2)[ids.reshape(-1)[perm]].astype(np.float64)[:, None]
        mask, alt = C.nvfp4_alternates(h * sc, rel)
        near = C.nvfp4_dequantize(*C.nvfp4_quantize((h * sc).astype(np.float32))) / sc
        alt = alt / sc
    elif a8:
        # with an activation global scale the decisions are taken on a2 * h
        sc = (np.ones(h.shape[0]) if a2 is None else
              np.float32(a2)[ids.reshape(-1)[perm]].astype(np.float64))[:, None]
        mask, alt = C.mxfp8_alternates(h * sc, rel)
        q, s = C.mxfp8_quantize(h * sc)
        near = C.mxfp8_dequantize(q, s) / sc
        alt = alt / sc
    else:
        mask, alt = C.bf16_alternates(h, rel)
        near = C.bf16_round(h)
        if kept_a8:
            # the kept tier's slots round h to static FP8 with the w2 input scale
            kept = np.array([kept_a8_scales(ck, int(e), True) is not None
                             for e in ids.reshape(-1)[perm]], dtype=bool)
            if kept.any():
                m8, a8v = C.fp8_static_alternates(h[kept], ck.in2, rel)
                mask[kept], alt[kept] = m8, a8v
                near[kept] = C.fp8_static_quantize(h[kept], ck.in2)[1]
    want = set(range(M)) if rows is None else set(int(r) for r in rows)
    out = {r: [] for r in want}
    cache = {}
    for p, i in zip(*np.nonzero(mask)):
        f = int(perm[p])
        t, j = divmod(f, k)
        if t not in want:
            continue
        e = int(ids[t, j])
        if e not in cache:
            cache[e] = expert_weights(ck, e)[1]
        cw = 1.0 if weight_on_input else w[t, j]
        out[t].append(cw * (alt[p, i] - near[p, i]) * cache[e][:, i])
    return out


def _fp8_static_scalar(v: float, s) -> float:
    """One value through static per-tensor FP8, by exhaustive search for the brute force:
    p = fp32(fp32(v) * fp32(1 / s)); the E4M3 magnitude nearest to min(|p|, 448) among the 127
    finite codes (ties to the even code); with p's sign, times s."""
    s32 = np.float32(s)
    p = float(np.float32(np.float32(v) * (np.float32(1.0) / s32)))
    mag = min(abs(p), 448.0)
    code = min(range(127), key=lambda c: (abs(C.e4m3_value(c) - mag), c % 2))
    return math.copysign(C.e4m3_value(code), p) * float(s32)


def moe_forward_bruteforce(ck, x_bits, topk_ids, topk_w, limit=math.inf, alpha=1.0, beta=0.0,
                           weight_on_input=False, fc2_override=None, return_f64=False,
                           kept_a8=False):
    """Token by token, slot by slot, element by element (pure Python loops; tiny inputs only).
    Dequantises each weight element from its own code and scale with scalar decoders.
    ``weight_on_input``: each input element becomes the bf16 rounding of x * bf16(w) and the
    slot's output is added unweighted.  ``fc2_override`` ({(t, j): {i: value}}) replaces
    element i of slot (t, j)'s fc2 operand (the dequantised intermediate) by the given value, so
    a test can take one rounding decision the other way.  Returns bf16 bit patterns (and the
    unrounded fp64 sums when ``return_f64``)."""
    ids = np.asarray(topk_ids).tolist()
    w = np.asarray(topk_w, dtype=np.float64).tolist()
    M = len(ids)
    E, H, I = ck.E, ck.H, ck.I
    a8 = activation_a8(ck)
    a1, a2 = act_gscale(ck, "a1"), act_gscale(ck, "a2")
    _, _, xhat = quantize_x(np.asarray(x_bits), a8 and a1 is None)
    out = [[0.0] * H for _ in range(M)]

    tiers = tier_local_index(ck.tier) if ck.quant == "hybrid" else None

    def weight(mat, e, r, c):
        """Scalar decode of element (r, c) of expert e's matrix ('w13' or 'w2')."""
        if tiers is not None:
            t, li = tiers[e]
            sub = ck.nv if t == TIER_NVFP4 else ck.nf
        else:
            sub, li = ck, e
        codes = getattr(sub, mat)[li]
        scales = getattr(sub, "s13" if mat == "w13" else "s2")[li]
        if sub.quant in ("mxfp4", "nvfp4", "w4a8_nvfp4", "w4a4_nvfp4"):
            byte = int(codes[r, c // 2])
            nib = byte & 0xF if c % 2 == 0 else byte >> 4
            v = C.e2m1_value(nib)
            if sub.quant == "mxfp4":
                return v * 2.0 ** (int(scales[r, c // 32]) - 127)
            g = float((sub.g13 if mat == "w13" else sub.g2)[li])
            return v * C.e4m3_value(int(scales[r, c // 16])) * g
        # NF3: bytes 3*(c//8) .. +2 hold codes c//8*8 .. +7
        b = codes[r, 3 * (c // 8): 3 * (c // 8) + 3]
        w24 = int(b[0]) | (int(b[1]) << 8) | (int(b[2]) << 16)
        code = (w24 >> (3 * (c % 8))) & 7
        prod = np.float32(C.NF3_LUT[code]) * np.float32(C.e4m3_value(int(scales[r, c // 32])))
        return float(C.bf16_round(float(prod)))

    for t in range(M):
        for j in range(len(ids[t])):
            e = ids[t][j]
            if not (0 <= e < E):
                continue
            xt = xhat[t]
            if activation_nv4(ck):
                xt = nvfp4_act(C.bf16_bits_to_f64(np.asarray(x_bits)[t:t + 1]), a1[e])[0]
            elif a1 is not None:
                xt = quantize_x(np.asarray(x_bits)[t:t + 1], True, a1[e])[2][0]
            s8 = kept_a8_scales(ck, e, kept_a8)
            if s8 is not None:
                xt = [_fp8_static_scalar(float(v), s8[0])
                      for v in C.bf16_bits_to_f64(np.asarray(x_bits)[t])]
            cw = w[t][j]
            if weight_on_input:
                wb = float(C.bf16_round(cw))
                xt = [float(C.bf16_round(float(v) * wb)) for v in xt]
                cw = 1.0
            gate = [0.0] * I
            up = [0.0] * I
            for i in range(I):
                up_row = i if ck.layout == W13_UP_GATE else I + i
                gate_row = I + i if ck.layout == W13_UP_GATE else i
                su = 0.0
                sg = 0.0
                for c in range(H):
                    su += weight("w13", e, up_row, c) * xt[c]
                    sg += weight("w13", e, gate_row, c) * xt[c]
                up[i] = su
                gate[i] = sg
            h = [0.0] * I
            for i in range(I):
                g = min(gate[i], limit)
                u = max(-limit, min(up[i], limit))
                h[i] = g * (1.0 / (1.0 + math.exp(-alpha * g))) * (u + beta)
            if s8 is not None:
                hh = [_fp8_static_scalar(v, s8[1]) for v in h]
            else:
                hh = (nvfp4_act(np.array(h)[None, :], a2[e])[0] if activation_nv4(ck) else
                      requant_h(np.array(h), a8, None if a2 is None else a2[e])).tolist()
            for i, v in ((fc2_override or {}).get((t, j)) or {}).items():
                hh[i] = float(v)
            for r in range(H):
                s = 0.0
                for i in range(I):
                    s += weight("w2", e, r, i) * hh[i]
                out[t][r] += cw * s
    bits = C.f64_to_bf16_bits(np.array(out))
    if return_f64:
        return bits, np.array(out)
    return bits


# ---------------------------------------------------------------------------- bounds

def _bf16_half_ulp(v):
    """Half the spacing of bf16 values in the binade of v (8 significant bits)."""
    _, ex = np.frexp(np.where(v == 0, 1.0, v))          # |v| in [2^(ex-1), 2^ex)
    return np.ldexp(1.0, np.maximum(ex.astype(np.int64) - 1, -126) - 8)


def row_errors(got_bits, ref_f64):
    """Per-row relative L2 error, and the largest error beyond the output's own rounding as a
    fraction of the row's rms, of bf16 output against the fp64 sum.

    The output is bf16, so even the exact result rounded once misses by up to half a bf16 ulp
    of each element; an element far above the row's rms (an outlier) would make that unavoidable
    rounding alone exceed a bound on max|err| / rms.  So the second figure measures
    max(|err| - half_ulp(ref), 0) / rms: it is 0 for the correctly rounded result and grows
    with any error of the computation.  A row whose reference is zero must be exactly zero."""
    got = C.bf16_bits_to_f64(got_bits)
    ref = np.asarray(ref_f64, dtype=np.float64)
    diff = got - ref
    nref = np.sqrt((ref ** 2).sum(axis=1))
    rms = np.sqrt((ref ** 2).mean(axis=1))
    rel = np.sqrt((diff ** 2).sum(axis=1)) / np.where(nref > 0, nref, 1.0)
    excess = np.maximum(np.abs(diff) - _bf16_half_ulp(ref), 0.0)
    mx = excess.max(axis=1) / np.where(rms > 0, rms, 1.0)
    zero_rows = nref == 0
    rel[zero_rows] = np.where(np.abs(got[zero_rows]).max(axis=1) == 0, 0.0, np.inf) \
        if zero_rows.any() else rel[zero_rows]
    mx[zero_rows] = rel[zero_rows]
    return rel, mx
