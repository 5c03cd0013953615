"""Routed MoE FFN layer on one B300: thin Python binding of the C ABI in include/moe.h (and moe_gen.h).

Every function here only marshals arguments (torch tensors or integer device pointers, streams)
into the C entry points of ``libmoe_b300.so``; all computation runs in the library's CUDA kernels.
Importing this package fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_OOM",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_NOT_SET", 7: "MOE_ERR_DEVICE"}
MOE_ACT_F32, MOE_ACT_BF16 = 0, 1
MOE_W_F32, MOE_W_INT4_G32 = 0, 1
SMALL_T = 16  # T <= SMALL_T can run the split-K GEMV path
MOE_OPT_GEMV_MAX_TOKENS = 1
MOE_OPT_FUSED_MAX_TOKENS = 2
MOE_OPT_KERNEL_TIMELINE = 3
TIMELINE_EVENTS = ("start", "dep_wait", "logits", "unit_computed", "routed", "first_unit", "units_done", "first_down",
                   "down_done", "end", "last_unit_issued", "first_down_issued", "last_down_issued",
                   "first_unit_issued", "clk_start", "clk_end", "x_staged", "router_rows", "keys", "selected",
                   "dispatched", "producer_routed", "unit_reduced", "first_down_done", "producer_go",
                   "gather_start", "first_routed_landed", "first_routed_done", "last_down_done",
                   "second_landed", "second_computed", "second_done")


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = f"{fn} returned {STATUS_NAMES.get(status, status)}"
        if status == 4:
            code = lib.moe_last_cuda_error()
            msg += f" (CUDA error {code}: {lib.moe_cuda_error_string(code).decode()})"
        super().__init__(msg)


class moe_config(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("f", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("n_layers", ctypes.c_int), ("max_tokens", ctypes.c_int), ("has_shared", ctypes.c_int),
                ("prenorm", ctypes.c_int), ("norm_eps", ctypes.c_float), ("wfmt", ctypes.c_int),
                ("act", ctypes.c_int)]


class moe_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("router_w", "router_b", "gu_q", "gu_s", "dn_q", "dn_s",
                                                "sh_gu_q", "sh_gu_s", "sh_dn_q", "sh_dn_s")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} is missing "
                          "(run `python -m routed_expert_ffn_07_b300.build`)")
    L = ctypes.CDLL(LIB_PATH)
    vp, ci, i32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    sig = {
        "moe_create": ([ctypes.POINTER(moe_config), ctypes.POINTER(vp)], ci),
        "moe_set_layer": ([vp, ci, ctypes.POINTER(moe_layer_weights)], ci),
        "moe_route": ([vp, ci, vp, ci, i32p, vp, i32p, i32p, vp], ci),
        "moe_layer_forward": ([vp, ci, vp, ci, vp, vp], ci),
        "moe_stack_forward": ([vp, vp, ci, vp, vp], ci),
        "moe_stack_forward_traced": ([vp, vp, ci, vp, i32p, vp, i32p, i32p, vp], ci),
        "moe_get_last_routing": ([vp, ci, i32p, vp, i32p, i32p, vp], ci),
        "moe_usage_enable": ([vp, ci], ci),
        "moe_usage_read": ([vp, vp, ci, vp], ci),
        "moe_layer_forward_host": ([vp, ci, vp, ci, vp, vp], ci),
        "moe_get_active_counts": ([vp, i32p, vp], ci),
        "moe_get_device_status": ([vp, vp], ci),
        "moe_destroy": ([vp], ci),
        "moe_route_noalloc": ([vp, vp, vp, ci, ci, ci, ci, ci, i32p, vp, i32p, i32p, vp], ci),
        "moe_set_option": ([vp, ci, ci], ci),
        "moe_selftest_bounded_waits": ([ctypes.c_longlong, vp], ci),
        "moe_inject_device_status": ([vp, ctypes.c_uint, vp], ci),
        "moe_timing_enable": ([vp, ci], ci),
        "moe_timing_rewind": ([vp], ci),
        "moe_timing_read": ([vp, vp, ci, ctypes.POINTER(ci), vp], ci),
        "moe_timeline_read": ([vp, vp, ci, ctypes.POINTER(ci), ctypes.POINTER(ci), vp], ci),
        "moe_status_str": ([ci], ctypes.c_char_p),
        "moe_version": ([], ci),
        "moe_last_cuda_error": ([], ci),
        "moe_peek_cuda_error": ([], ci),
        "moe_cuda_error_string": ([ci], ctypes.c_char_p),
        "moe_gen_int4_planes": ([vp, ctypes.c_uint64, ci, ci, ci, ci, ctypes.c_size_t, vp], ci),
        "moe_gen_scale_planes": ([vp, ctypes.c_uint64, ci, ci, ci, ci, ctypes.c_size_t, vp], ci),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


lib = _load()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _check(fn, st):
    if st != MOE_OK:
        raise MoeError(fn, st)


def moe_create(d, f, n_experts, top_k, n_layers, max_tokens, has_shared=True, prenorm=False, norm_eps=1e-6,
               wfmt=MOE_W_INT4_G32, act=MOE_ACT_BF16):
    cfg = moe_config(d, f, n_experts, top_k, n_layers, max_tokens, int(has_shared), int(prenorm),
                     float(norm_eps), wfmt, act)
    h = ctypes.c_void_p()
    _check("moe_create", lib.moe_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def moe_set_layer(h, layer, router_w, gu_q, gu_s, dn_q, dn_s, router_b=None, sh_gu_q=None, sh_gu_s=None,
                  sh_dn_q=None, sh_dn_s=None):
    w = moe_layer_weights(*[_ptr(p) for p in (router_w, router_b, gu_q, gu_s, dn_q, dn_s,
                                              sh_gu_q, sh_gu_s, sh_dn_q, sh_dn_s)])
    _check("moe_set_layer", lib.moe_set_layer(h, layer, ctypes.byref(w)))


def moe_route(h, layer, x, T, topk_idx=None, topk_w=None, expert_offs=None, perm=None, stream=None):
    _check("moe_route", lib.moe_route(h, layer, _ptr(x), T, _ptr(topk_idx), _ptr(topk_w), _ptr(expert_offs),
                                      _ptr(perm), _stream(stream)))


def moe_route_noalloc(router_w, router_b, x, act, T, d, E, K, topk_idx=None, topk_w=None, expert_offs=None,
                      perm=None, stream=None):
    """Routing that allocates nothing (fixed device scratch inside the library); see include/moe.h."""
    _check("moe_route_noalloc", lib.moe_route_noalloc(_ptr(router_w), _ptr(router_b), _ptr(x), act, T, d, E, K,
                                                      _ptr(topk_idx), _ptr(topk_w), _ptr(expert_offs), _ptr(perm),
                                                      _stream(stream)))


def moe_layer_forward(h, layer, x, T, y, stream=None):
    _check("moe_layer_forward", lib.moe_layer_forward(h, layer, _ptr(x), T, _ptr(y), _stream(stream)))


def moe_stack_forward(h, x_inout, T, trace=None, stream=None):
    _check("moe_stack_forward", lib.moe_stack_forward(h, _ptr(x_inout), T, _ptr(trace), _stream(stream)))


def moe_stack_forward_traced(h, x_inout, T, trace=None, route_idx=None, route_w=None, route_offs=None,
                             route_perm=None, stream=None):
    _check("moe_stack_forward_traced",
           lib.moe_stack_forward_traced(h, _ptr(x_inout), T, _ptr(trace), _ptr(route_idx), _ptr(route_w),
                                        _ptr(route_offs), _ptr(route_perm), _stream(stream)))


def moe_get_last_routing(h, T, topk_idx=None, topk_w=None, expert_offs=None, perm=None, stream=None):
    _check("moe_get_last_routing", lib.moe_get_last_routing(h, T, _ptr(topk_idx), _ptr(topk_w), _ptr(expert_offs),
                                                            _ptr(perm), _stream(stream)))


def moe_usage_enable(h, on=True):
    _check("moe_usage_enable", lib.moe_usage_enable(h, int(bool(on))))


def moe_usage_read(h, n_layers, n_experts, reset=False, stream=None):
    """The per-layer expert usage histogram as a uint64 array [n_layers, n_experts]."""
    import numpy as np
    out = np.zeros((n_layers, n_experts), dtype=np.uint64)
    _check("moe_usage_read", lib.moe_usage_read(h, out.ctypes.data, int(bool(reset)), _stream(stream)))
    return out


def moe_layer_forward_host(h, layer, x_host, T, y_host, stream=None):
    _check("moe_layer_forward_host",
           lib.moe_layer_forward_host(h, layer, _ptr(x_host), T, _ptr(y_host), _stream(stream)))


def moe_get_active_counts(h, n_layers, stream=None):
    import numpy as np
    out = np.zeros(n_layers, dtype=np.int32)
    _check("moe_get_active_counts", lib.moe_get_active_counts(h, out.ctypes.data, _stream(stream)))
    return out


def moe_get_device_status(h, stream=None):
    return lib.moe_get_device_status(h, _stream(stream))


def moe_destroy(h):
    _check("moe_destroy", lib.moe_destroy(h))


def moe_inject_device_status(h, bits, stream=None):
    """Test hook: OR `bits` into the handle's device status word (see include/moe.h)."""
    _check("moe_inject_device_status", lib.moe_inject_device_status(h, bits, _stream(stream)))


def moe_selftest_bounded_waits(budget_cycles=2_000_000, stream=None):
    """Run the device self-test of the bounded waits; returns the raw moe_status (5 = timeout, expected)."""
    return lib.moe_selftest_bounded_waits(budget_cycles, _stream(stream))


def moe_set_option(h, option, value):
    r = lib.moe_set_option(h, option, value)
    if r < 0:
        raise MoeError("moe_set_option", -r)
    return r


def moe_timing_enable(h, n_records):
    _check("moe_timing_enable", lib.moe_timing_enable(h, n_records))


def moe_timing_rewind(h):
    _check("moe_timing_rewind", lib.moe_timing_rewind(h))


def moe_timing_read(h, max_records, stream=None):
    """Returns a float32 array [n_records, 4] of (route, stage A, stage B, stage C) milliseconds."""
    import numpy as np
    ms = np.zeros((max(max_records, 1), 4), dtype=np.float32)
    n = ctypes.c_int(0)
    _check("moe_timing_read", lib.moe_timing_read(h, ms.ctypes.data, max_records, ctypes.byref(n), _stream(stream)))
    return ms[: n.value].copy()


def moe_timeline_read(h, stream=None):
    """The one-launch decode layer's most recent in-kernel timeline: uint64 [n_ctas, n_events] (ns)."""
    import numpy as np
    cap = 4096 * 16
    out = np.zeros(cap, dtype=np.uint64)
    nc, ne = ctypes.c_int(0), ctypes.c_int(0)
    _check("moe_timeline_read", lib.moe_timeline_read(h, out.ctypes.data, cap, ctypes.byref(nc), ctypes.byref(ne),
                                                      _stream(stream)))
    return out[: nc.value * ne.value].reshape(nc.value, ne.value).copy()


def moe_status_str(s):
    return lib.moe_status_str(s).decode()


def moe_version():
    return lib.moe_version()


def moe_gen_int4_planes(dst, seed, layer, tensor, expert0, n_experts, bytes_per_expert, stream=None):
    rc = lib.moe_gen_int4_planes(_ptr(dst), seed, layer, tensor, expert0, n_experts, bytes_per_expert,
                                 _stream(stream))
    if rc:
        raise RuntimeError(f"moe_gen_int4_planes failed ({rc})")


def moe_gen_scale_planes(dst, seed, layer, tensor, expert0, n_experts, scales_per_expert, stream=None):
    rc = lib.moe_gen_scale_planes(_ptr(dst), seed, layer, tensor, expert0, n_experts, scales_per_expert,
                                  _stream(stream))
    if rc:
        raise RuntimeError(f"moe_gen_scale_planes failed ({rc})")
