"""Shared helpers of the GPU tests: build a layer from a synth checkpoint, run it through the
C ABI and compare with the oracle on the same seeded inputs."""
import math

import numpy as np

from oracle import codecs as C
from oracle import moe as O
from synth import moe_inputs as S

REL_L2_BOUND = 5e-3       # per-row relative L2 error
MAX_ERR_BOUND = 2e-2      # per-row max |err| / rms(row)


def to_device(x_bits, ids, w):
    import torch
    xt = torch.from_numpy(x_bits.view(np.int16).copy()).view(torch.bfloat16).cuda()
    it = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    wt = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    return xt, it, wt


def out_bits(out):
    return out.view(dtype=__import__("torch").int16).cpu().numpy().view(np.uint16)


def run_layer(layer, x_bits, ids, w):
    xt, it, wt = to_device(x_bits, ids, w)
    out = layer(xt, it, wt)
    return out_bits(out)


REQUANT_REL = 1e-4       # relative window of a rounding decision taken in fp32 arithmetic
# absolute part of the intermediate's ambiguity window, as a fraction of the slot's rms: a gate
# or up sum that cancels keeps the absolute fp32 error of its terms (about 2^-24 * sqrt(K) of
# their size), so an element far smaller than the slot's rms can sit that close to a midpoint
H_CANCEL_ATOL = 2.0 ** -16


def _row_ok(got_row_bits, ref_row):
    rel, mx = O.row_errors(got_row_bits[None, :], ref_row[None, :])
    return rel[0] <= REL_L2_BOUND and mx[0] <= MAX_ERR_BOUND, rel[0], mx[0]


def oracle_rows(ck, x_bits, ids, w, limit, rows=None, alpha=1.0, beta=0.0,
                weight_on_input=False, kept_a8=False):
    """The oracle's unrounded fp64 output for the given rows (all when None), to be shared by
    several check_rows calls on the same inputs."""
    rows = np.arange(ids.shape[0]) if rows is None else np.asarray(rows)
    _, f64 = O.moe_forward(ck, x_bits, ids, w, limit, alpha, beta, rows=rows, return_f64=True,
                           weight_on_input=weight_on_input, kept_a8=kept_a8)
    return f64


def check_rows(got_bits, ck, x_bits, ids, w, limit, rows=None, alpha=1.0, beta=0.0,
               weight_on_input=False, ref_f64=None, kept_a8=False):
    """Compare the given rows (all when None) with the oracle; returns (rel, mx) arrays.
    ``ref_f64``: the oracle's output of these inputs when already computed (oracle_rows).

    A row that misses the bound passes if the oracle's own alternatives of near-midpoint
    requantisation decisions (oracle.moe.requant_alternatives; any subset of up to 10 of them)
    bring it within the bound: those elements are decided by fp32 noise, both roundings are
    correct results of the method."""
    rows = np.arange(ids.shape[0]) if rows is None else np.asarray(rows)
    f64 = ref_f64 if ref_f64 is not None else oracle_rows(
        ck, x_bits, ids, w, limit, rows, alpha, beta, weight_on_input, kept_a8)
    rel, mx = O.row_errors(got_bits[rows], f64[rows])
    bad = [int(r) for r, a, b in zip(rows, rel, mx) if a > REL_L2_BOUND or b > MAX_ERR_BOUND]
    if bad:
        alts = O.requant_alternatives(ck, x_bits, ids, w, limit, alpha, beta, REQUANT_REL, bad,
                                      weight_on_input, kept_a8)
        for r in bad:
            d = alts[r]
            assert 0 < len(d) <= 10, (r, "outside the bound with", len(d), "ambiguous elements",
                                      O.row_errors(got_bits[[r]], f64[[r]]))
            ok = False
            for m in range(1, 1 << len(d)):
                ref = f64[r] + sum(d[i] for i in range(len(d)) if m >> i & 1)
                if _row_ok(got_bits[r], ref)[0]:
                    ok = True
                    break
            assert ok, (r, O.row_errors(got_bits[[r]], f64[[r]]))
    valid = ((ids >= 0) & (ids < ck.E)).any(axis=1)
    for r in rows:
        if not valid[r]:
            assert np.all(got_bits[r] == 0), r
    return rel, mx


def small_cfg(quant, E=16, H=1280, I=192, topk=4, n_nvfp4=5):
    base = {"mxfp4": S.CONFIGS["tiny_w4a8"], "nvfp4": S.CONFIGS["w4a16_nvfp4"],
            "hybrid": S.CONFIGS["hybrid_nvfp4_nf3"],
            "hybrid_mx": S.CONFIGS["hybrid_mxfp4_nf3"],
            "w4a8_nvfp4": S.CONFIGS["w4a8_nvfp4"], "w4a4_nvfp4": S.CONFIGS["w4a4_nvfp4"]}[quant]
    d = dict(base.__dict__)
    d.update(E=E, H=H, I=I, topk=topk, n_nvfp4=min(n_nvfp4, E))
    return S.MoEConfig(**d)
