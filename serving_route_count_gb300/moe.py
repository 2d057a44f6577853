"""Python binding of the C ABI (include/moe_gb300.h): argument marshalling only.

Every function has the name of the C entry point it calls.  Device buffers are torch CUDA
tensors (torch is used for device memory and streams only); every step of the computation
runs in the library's CUDA kernels.  There is no CPU fallback: a missing library raises.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib

MOE_W4A8_MXFP4 = 0
MOE_W4A16_NVFP4 = 1
MOE_W4A16_HYBRID = 2
MOE_W4A16_HYBRID_MX = 3
MOE_W4A8_NVFP4 = 4
MOE_W4A4_NVFP4 = 5
MOE_W13_UP_GATE = 0
MOE_W13_GATE_UP = 1
MOE_TIER_NVFP4 = 4
MOE_TIER_NF3 = 3

STATUS = {0: "MOE_OK", 1: "MOE_ERR_ARG", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_UNSUPPORTED",
          4: "MOE_ERR_CAPACITY", 5: "MOE_ERR_CAPTURING", 6: "MOE_ERR_CUDA", 7: "MOE_ERR_TIMEOUT",
          8: "MOE_ERR_DEVICE"}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def _check(st: int, where: str):
    if st != 0:
        if st == 6:   # MOE_ERR_CUDA: name the CUDA error behind it
            where = f"{where} ({_lib.load().moe_last_cuda_error().decode()})"
        raise MoEError(st, where)


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            raise ValueError("tensors passed to the library must be contiguous")
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        if not t.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays passed to the library must be C-contiguous")
        return t.ctypes.data
    return int(t)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _handle(h) -> ctypes.c_void_p:
    return ctypes.c_void_p(h)


# ---------------------------------------------------------------------------------- planning

def moe_plan_weights(E, H, I, quant_mode, w13_layout=MOE_W13_UP_GATE, tier_of_expert=None) -> int:
    L = _lib.load()
    out = ctypes.c_void_p()
    tier_p = None
    if tier_of_expert is not None:
        tier = np.ascontiguousarray(np.asarray(tier_of_expert, dtype=np.int8))
        tier_p = tier.ctypes.data_as(_lib.c_int8_p)
    _check(L.moe_plan_weights(E, H, I, quant_mode, w13_layout, tier_p, ctypes.byref(out)),
           "moe_plan_weights")
    return out.value


def moe_prepared_bytes(wp) -> int:
    n = ctypes.c_size_t()
    _check(_lib.load().moe_prepared_bytes(_handle(wp), ctypes.byref(n)), "moe_prepared_bytes")
    return n.value


def moe_prepare_weights(wp, ckpt: dict, dst: torch.Tensor, stream=None) -> int:
    """ckpt: dict of device tensors keyed like moe_checkpoint's fields (missing keys = NULL)."""
    c = _lib.MoeCheckpoint(*[_ptr(ckpt.get(f)) or None for f, _ in _lib.MoeCheckpoint._fields_])
    out = ctypes.c_void_p()
    _check(_lib.load().moe_prepare_weights(_handle(wp), ctypes.byref(c), _ptr(dst),
                                           dst.numel() * dst.element_size(), _stream(stream),
                                           ctypes.byref(out)), "moe_prepare_weights")
    return out.value


def moe_unprepare_weights(wp, prepared, like: dict, stream=None) -> dict:
    """Test hook: checkpoint-layout host arrays of prepared weights.  ``like`` maps the
    moe_checkpoint field names to numpy arrays giving each output's shape and dtype (missing
    fields stay NULL)."""
    out = {k: np.zeros_like(v) for k, v in like.items() if v is not None}
    c = _lib.MoeCheckpoint(*[(out[f].ctypes.data if f in out else None)
                             for f, _ in _lib.MoeCheckpoint._fields_])
    _check(_lib.load().moe_unprepare_weights(_handle(wp), _handle(prepared), _stream(stream),
                                             ctypes.byref(c)), "moe_unprepare_weights")
    return out


def moe_plan(E, H, I, topk, max_m, quant_mode, swiglu_limit=float("inf"), deterministic=0) -> int:
    out = ctypes.c_void_p()
    _check(_lib.load().moe_plan(E, H, I, topk, max_m, quant_mode, float(swiglu_limit),
                                int(bool(deterministic)), ctypes.byref(out)), "moe_plan")
    return out.value


def moe_plan_set_swiglu_alpha_beta(plan, alpha, beta):
    _check(_lib.load().moe_plan_set_swiglu_alpha_beta(_handle(plan), float(alpha), float(beta)),
           "moe_plan_set_swiglu_alpha_beta")


def moe_plan_set_backend(plan, backend):
    _check(_lib.load().moe_plan_set_backend(_handle(plan), int(backend)), "moe_plan_set_backend")


def moe_plan_set_fc1_kernel(plan, choice):
    _check(_lib.load().moe_plan_set_fc1_kernel(_handle(plan), int(choice)),
           "moe_plan_set_fc1_kernel")


def moe_plan_set_router_weight_on_input(plan, on):
    _check(_lib.load().moe_plan_set_router_weight_on_input(_handle(plan), int(on)),
           "moe_plan_set_router_weight_on_input")


def moe_plan_set_expert_offset(plan, first_expert):
    _check(_lib.load().moe_plan_set_expert_offset(_handle(plan), int(first_expert)),
           "moe_plan_set_expert_offset")


def moe_scratch_bytes(plan) -> int:
    n = ctypes.c_size_t()
    _check(_lib.load().moe_scratch_bytes(_handle(plan), ctypes.byref(n)), "moe_scratch_bytes")
    return n.value


def moe_io_bytes(plan) -> int:
    n = ctypes.c_size_t()
    _check(_lib.load().moe_io_bytes(_handle(plan), ctypes.byref(n)), "moe_io_bytes")
    return n.value


# ---------------------------------------------------------------------------------- running

def moe_run(plan, prepared, scratch: torch.Tensor, x, topk_ids, topk_weights, out, M=None,
            stream=None):
    M = x.shape[0] if M is None else M
    _check(_lib.load().moe_run(_handle(plan), _handle(prepared), _ptr(scratch),
                               scratch.numel() * scratch.element_size(), _ptr(x), _ptr(topk_ids),
                               _ptr(topk_weights), _ptr(out), int(M), _stream(stream)), "moe_run")


def moe_run_chunked(plan, prepared, scratch: torch.Tensor, x, topk_ids, topk_weights, out,
                    M=None, stream=None):
    """moe_run for any number of rows: chunks of the plan's capacity, run in order."""
    M = x.shape[0] if M is None else M
    _check(_lib.load().moe_run_chunked(_handle(plan), _handle(prepared), _ptr(scratch),
                                       scratch.numel() * scratch.element_size(), _ptr(x),
                                       _ptr(topk_ids), _ptr(topk_weights), _ptr(out), int(M),
                                       _stream(stream)), "moe_run_chunked")


def moe_run_static_scratch(plan, prepared, x, topk_ids, topk_weights, out, M=None, stream=None):
    """moe_run with the scratch in the library's fixed 16 MiB device array, for callers that
    cannot allocate device memory (see include/moe_gb300.h).  Calls on one device share that
    array: overlapping calls must be serialised by the caller."""
    M = x.shape[0] if M is None else M
    _check(_lib.load().moe_run_static_scratch(_handle(plan), _handle(prepared), _ptr(x),
                                              _ptr(topk_ids), _ptr(topk_weights), _ptr(out),
                                              int(M), _stream(stream)), "moe_run_static_scratch")


def moe_run_host(plan, prepared, scratch, io, x_host, ids_host, w_host, out_host, M=None,
                 stream=None):
    M = x_host.shape[0] if M is None else M
    _check(_lib.load().moe_run_host(_handle(plan), _handle(prepared), _ptr(scratch),
                                    scratch.numel() * scratch.element_size(), _ptr(io),
                                    io.numel() * io.element_size(), _ptr(x_host), _ptr(ids_host),
                                    _ptr(w_host), _ptr(out_host), int(M), _stream(stream)),
           "moe_run_host")


def moe_get_device_error(plan, scratch, stream=None):
    code = ctypes.c_int()
    st = _lib.load().moe_get_device_error(_handle(plan), _ptr(scratch), _stream(stream),
                                          ctypes.byref(code))
    return st, code.value


def moe_plan_set_kept_a8(plan, w13_input_scale, w2_input_scale):
    _check(_lib.load().moe_plan_set_kept_a8(_handle(plan), float(w13_input_scale),
                                            float(w2_input_scale)), "moe_plan_set_kept_a8")


def moe_plan_set_wait_probe(plan, ns):
    _check(_lib.load().moe_plan_set_wait_probe(_handle(plan), int(ns)), "moe_plan_set_wait_probe")


def moe_plan_set_debug_copies(plan, on):
    _check(_lib.load().moe_plan_set_debug_copies(_handle(plan), int(on)),
           "moe_plan_set_debug_copies")


def moe_get_device_error_static(plan, stream=None):
    """moe_get_device_error for calls made with moe_run_static_scratch: (status, code)."""
    code = ctypes.c_int()
    st = _lib.load().moe_get_device_error_static(_handle(plan), _stream(stream),
                                                 ctypes.byref(code))
    return st, code.value


def moe_debug_routing(plan, scratch, M, E, topk, stream=None):
    cnt = np.zeros(E, np.int32)
    off = np.zeros(E + 1, np.int32)
    perm = np.zeros(max(1, M * topk), np.int32)
    slot_of = np.zeros(max(1, M * topk), np.int32)
    _check(_lib.load().moe_debug_routing(_handle(plan), _ptr(scratch), int(M), _ptr(cnt),
                                         _ptr(off), _ptr(perm), _ptr(slot_of), _stream(stream)),
           "moe_debug_routing")
    return cnt, off, perm[: off[E]], slot_of[: M * topk]


def moe_debug_actq(plan, scratch, M, H, topk, stream=None):
    """Quantised activations in slot order: row p is the MXFP8 row of token perm[p] // topk."""
    xq = np.zeros((max(1, M * topk), H), np.uint8)
    xs = np.zeros((max(1, M * topk), H // 32), np.uint8)
    _check(_lib.load().moe_debug_actq(_handle(plan), _ptr(scratch), int(M), _ptr(xq), _ptr(xs),
                                      _stream(stream)), "moe_debug_actq")
    return xq, xs


def moe_debug_h(plan, scratch, M, Ip, topk, a8, stream=None, a4=False):
    """fc2 activation operand of the last call in slot order: (codes, scales) for W4A8,
    (packed E2M1 codes [rows][Ip/2], E4M3 scales [rows][Ip/16]) for W4A4, (f16 bits, None)
    otherwise."""
    rows = max(1, M * topk)
    if a4:
        hq = np.zeros((rows, Ip // 2), np.uint8)
        hs = np.zeros((rows, Ip // 16), np.uint8)
    elif a8:
        hq = np.zeros((rows, Ip), np.uint8)
        hs = np.zeros((rows, Ip // 32), np.uint8)
    else:
        hq = np.zeros((rows, Ip), np.uint16)
        hs = None
    _check(_lib.load().moe_debug_h(_handle(plan), _ptr(scratch), int(M), _ptr(hq), _ptr(hs),
                                   _stream(stream)), "moe_debug_h")
    return hq, hs


def moe_plan_set_profile_events(plan, events):
    """events: list of torch.cuda.Event(enable_timing=True) (or raw handles); [] turns it off."""
    hs = [ev.cuda_event if hasattr(ev, "cuda_event") else int(ev) for ev in events]
    arr = (ctypes.c_void_p * max(1, len(hs)))(*hs)
    _check(_lib.load().moe_plan_set_profile_events(_handle(plan), arr, len(hs)),
           "moe_plan_set_profile_events")


def moe_call_launches(plan, M) -> int:
    """Kernel launches moe_run makes for a call of M tokens."""
    n = ctypes.c_int(0)
    _check(_lib.load().moe_call_launches(_handle(plan), int(M), ctypes.byref(n)),
           "moe_call_launches")
    return n.value


def moe_profile_stage_names(plan):
    return _lib.load().moe_profile_stage_names(_handle(plan)).decode().split(",")


def moe_destroy_weight_plan(wp):
    _lib.load().moe_destroy_weight_plan(_handle(wp))


def moe_destroy_prepared(p):
    _lib.load().moe_destroy_prepared(_handle(p))


def moe_destroy_plan(plan):
    _lib.load().moe_destroy_plan(_handle(plan))


def moe_status_str(s) -> str:
    return _lib.load().moe_status_str(int(s)).decode()


def moe_version() -> str:
    return _lib.load().moe_version().decode()


# ---------------------------------------------------------------------------------- convenience

QUANT_OF = {"mxfp4": MOE_W4A8_MXFP4, "nvfp4": MOE_W4A16_NVFP4, "hybrid": MOE_W4A16_HYBRID,
            "w4a8_nvfp4": MOE_W4A8_NVFP4, "w4a4_nvfp4": MOE_W4A4_NVFP4}


def quant_mode_of(ck) -> int:
    """Library quant mode of a host checkpoint: a hybrid layer whose kept tier is MXFP4 is the
    MXFP4-kept hybrid mode."""
    if ck.quant == "hybrid" and ck.nv is not None and ck.nv.quant == "mxfp4":
        return MOE_W4A16_HYBRID_MX
    return QUANT_OF[ck.quant]


def checkpoint_to_device(ck, device="cuda") -> dict:
    """Upload a host checkpoint (fields like synth.Checkpoint) as device tensors keyed like
    moe_checkpoint."""
    def t(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)
    if ck.quant == "hybrid":
        nv, nf = ck.nv, ck.nf
        return {"w13": t(nv.w13), "s13": t(nv.s13), "g13": t(nv.g13), "w2": t(nv.w2),
                "s2": t(nv.s2), "g2": t(nv.g2), "nf_w13": t(nf.w13), "nf_s13": t(nf.s13),
                "nf_w2": t(nf.w2), "nf_s2": t(nf.s2)}
    return {"w13": t(ck.w13), "s13": t(ck.s13), "g13": t(ck.g13), "w2": t(ck.w2),
            "s2": t(ck.s2), "g2": t(ck.g2), "a1_gscale": t(getattr(ck, "a13", None)),
            "a2_gscale": t(getattr(ck, "a2", None))}


class MoELayer:
    """One layer: weight plan + prepared weights + execution plan + scratch, all device-resident.

    ``ck`` is a host checkpoint (synth.Checkpoint-like: quant, E, H, I, layout, tensors).
    """

    def __init__(self, ck, topk, max_m, swiglu_limit=float("inf"), deterministic=False,
                 alpha=None, beta=None, device="cuda", keep_checkpoint=False, backend=0,
                 fc1_kernel=0, first_expert=0, weight_on_input=False, debug_copies=False,
                 kept_a8=None):
        self.E, self.H, self.I, self.topk, self.max_m = ck.E, ck.H, ck.I, topk, max_m
        self.quant = quant_mode_of(ck)
        tier = ck.tier if ck.quant == "hybrid" else None
        self.wp = moe_plan_weights(ck.E, ck.H, ck.I, self.quant, ck.layout, tier)
        dev_ck = checkpoint_to_device(ck, device)
        self.wbuf = torch.empty(moe_prepared_bytes(self.wp), dtype=torch.uint8, device=device)
        self.prep = moe_prepare_weights(self.wp, dev_ck, self.wbuf)
        if not keep_checkpoint:
            torch.cuda.current_stream().synchronize()
            del dev_ck
        else:
            self.dev_ck = dev_ck
        self.plan = moe_plan(ck.E, ck.H, ck.I, topk, max_m, self.quant, swiglu_limit, deterministic)
        if alpha is not None or beta is not None:
            moe_plan_set_swiglu_alpha_beta(self.plan, 1.0 if alpha is None else alpha,
                                           0.0 if beta is None else beta)
        if backend:
            moe_plan_set_backend(self.plan, backend)
        if fc1_kernel:
            moe_plan_set_fc1_kernel(self.plan, fc1_kernel)
        if first_expert:
            moe_plan_set_expert_offset(self.plan, first_expert)
        if weight_on_input:
            moe_plan_set_router_weight_on_input(self.plan, 1)
        if debug_copies:
            moe_plan_set_debug_copies(self.plan, 1)
        if kept_a8 is not None:        # (w13_input_scale, w2_input_scale)
            moe_plan_set_kept_a8(self.plan, kept_a8[0], kept_a8[1])
        self.scratch = torch.empty(moe_scratch_bytes(self.plan), dtype=torch.uint8, device=device)
        self.device = device
        self._io = None

    def __call__(self, x, topk_ids, topk_weights, out=None, stream=None):
        if out is None:
            out = torch.empty((x.shape[0], self.H), dtype=torch.bfloat16, device=x.device)
        moe_run(self.plan, self.prep, self.scratch, x, topk_ids, topk_weights, out, stream=stream)
        return out

    def run_host(self, x_host, ids_host, w_host, out_host, stream=None):
        """moe_run_host on this layer; the layer's own arguments (plan, weights, scratch, staging
        buffer) are marshalled once, the host tensors on every call."""
        if self._io is None:
            self._io = torch.empty(moe_io_bytes(self.plan), dtype=torch.uint8, device=self.device)
            self._host_args = (_handle(self.plan), _handle(self.prep), _ptr(self.scratch),
                               self.scratch.numel(), _ptr(self._io), self._io.numel())
        for t in (x_host, ids_host, w_host, out_host):
            if not t.is_contiguous():
                raise ValueError("tensors passed to the library must be contiguous")
        _check(_lib.load().moe_run_host(*self._host_args, x_host.data_ptr(), ids_host.data_ptr(),
                                        w_host.data_ptr(), out_host.data_ptr(), x_host.shape[0],
                                        _stream(stream)), "moe_run_host")
        return out_host

    def routing(self, M, stream=None):
        return moe_debug_routing(self.plan, self.scratch, M, self.E, self.topk, stream)

    def actq(self, M, stream=None):
        """(xq, xs) of the last call in slot order, trimmed to the S valid slots."""
        S = int(self.routing(M, stream)[1][-1])
        xq, xs = moe_debug_actq(self.plan, self.scratch, M, self.H, self.topk, stream)
        return xq[:S], xs[:S]

    def intermediate(self, M, stream=None):
        """fc2 activation operand of the last call, trimmed to the S valid slots."""
        S = int(self.routing(M, stream)[1][-1])
        Ip = (self.I + 127) // 128 * 128
        hq, hs = moe_debug_h(self.plan, self.scratch, M, Ip, self.topk,
                             self.quant == MOE_W4A8_MXFP4, stream, self.quant == MOE_W4A4_NVFP4)
        return hq[:S], (hs[:S] if hs is not None else None)

    def device_error(self, stream=None):
        return moe_get_device_error(self.plan, self.scratch, stream)

    def close(self):
        if getattr(self, "plan", None):
            moe_destroy_plan(self.plan)
            self.plan = None
        if getattr(self, "prep", None):
            moe_destroy_prepared(self.prep)
            self.prep = None
        if getattr(self, "wp", None):
            moe_destroy_weight_plan(self.wp)
            self.wp = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
