"""ctypes binding of ``include/moe.h`` (libmoe.so): same names, argument marshalling only.

Device buffers are passed as torch CUDA tensors (or raw integer addresses);
streams as ``torch.cuda.Stream`` or a raw ``cudaStream_t`` integer (default: the
current torch stream).  A non-OK status raises :class:`MoeError`; nothing here
computes anything of the method, and importing this module fails loudly when
the library has not been built.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmoe.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} has not been built; run block_quantised_moe_gb300.build.build() "
        "(or __graft_entry__.build()) first")
_lib = ctypes.CDLL(_LIB_PATH)
LIB_PATH = _LIB_PATH

# ------------------------------------------------------------- constants
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CAPACITY = 0, 1, 2, 3
MOE_ERR_SCRATCH_TOO_SMALL, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = 4, 5, 6
MOE_W_NVFP4, MOE_W_MXFP4 = 1, 2
MOE_A_BF16, MOE_A_NVFP4, MOE_A_MXFP8 = 1, 2, 3
MOE_WFLAG_FP4_TILES = 1
MOE_ACT_SILU_GATED, MOE_ACT_RELU2 = 1, 2
MOE_Q_NVFP4, MOE_Q_MXFP4, MOE_Q_MXFP8 = 1, 2, 3
MOE_G_NONE, MOE_G_PER_TENSOR, MOE_G_PER_ROW = 0, 1, 2
MOE_NUM_STAGES = 6
STAGES = ("route", "quant_x", "gemm1", "quant_h", "gemm2", "combine")
MOE_NO_ALLOC_SCRATCH_BYTES = 32 << 20
MOE_OPT_SINGLE_LAUNCH = 1
MOE_OPT_OUT_F32 = 2

WFMT = {"nvfp4": MOE_W_NVFP4, "mxfp4": MOE_W_MXFP4}
AFMT = {"bf16": MOE_A_BF16, "nvfp4": MOE_A_NVFP4, "mxfp8": MOE_A_MXFP8}
ACT = {"silu": MOE_ACT_SILU_GATED, "relu2": MOE_ACT_RELU2}

# names exported by libmoe.so, as declared in include/moe.h
EXPORTS = (
    "moe_status_str", "moe_plan_weights", "moe_prepare_weights", "moe_is_supported", "moe_plan",
    "moe_bind", "moe_run", "moe_run_timed", "moe_run_host", "moe_device_status", "moe_debug_routing", "moe_quantize",
    "moe_destroy_weight_plan", "moe_destroy_plan", "moe_destroy_binding", "moe_run_no_alloc", "moe_launch_count",
    "moe_measure_mma_peak", "moe_selftest_wait_timeout", "moe_debug_hidden", "moe_no_alloc_device_status",
    "moe_plan_set_option", "moe_selftest_grid_barrier_timeout",
)


class moe_weight_desc(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("wfmt", ctypes.c_int32), ("act", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class moe_caps(ctypes.Structure):
    _fields_ = [("wplan", ctypes.c_void_p), ("top_k", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("afmt", ctypes.c_int32)]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_P = ctypes.POINTER
_sig = {
    "moe_status_str": (ctypes.c_char_p, [_i32]),
    "moe_plan_weights": (_i32, [_P(moe_weight_desc), _P(_vp), _P(_sz)]),
    "moe_prepare_weights": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_is_supported": (_i32, [_P(moe_caps)]),
    "moe_plan": (_i32, [_P(moe_caps), _P(_vp), _P(_sz), _P(_i32)]),
    "moe_bind": (_i32, [_vp, _vp, _sz, _vp, _vp, _vp, _vp, _i32, _vp, _P(_vp)]),
    "moe_run": (_i32, [_vp, _vp]),
    "moe_run_timed": (_i32, [_vp, _vp, _P(_vp)]),
    "moe_launch_count": (_i32, [_vp, _P(_i32)]),
    "moe_measure_mma_peak": (_i32, [_i32, _i32, _i32, _P(ctypes.c_float)]),
    "moe_run_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_device_status": (_i32, [_vp, _vp, _P(_i32)]),
    "moe_debug_routing": (_i32, [_vp, _vp, _P(_i32), _P(_i32), _P(_i32), _P(_i32), _i32]),
    "moe_quantize": (_i32, [_i32, _i32, _i32, _vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "moe_destroy_weight_plan": (None, [_vp]),
    "moe_destroy_plan": (None, [_vp]),
    "moe_destroy_binding": (None, [_vp]),
    "moe_run_no_alloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp]),
    "moe_no_alloc_device_status": (_i32, [_vp, _vp, _P(_i32)]),
    "moe_plan_set_option": (_i32, [_vp, _i32, _i32]),
    "moe_selftest_grid_barrier_timeout": (_i32, [_vp, _vp, _P(_i32)]),
    "moe_selftest_wait_timeout": (_i32, [_vp, _vp, _P(_i32)]),
    "moe_debug_hidden": (_i32, [_vp, _vp, _P(ctypes.c_float), _i32, _P(_i32)]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype, _f.argtypes = _res, _args


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {moe_status_str(status)}")


def moe_status_str(status: int) -> str:
    return _lib.moe_status_str(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(x):
    """Device or host address of a tensor / array / int; None -> NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------------ calls


def moe_plan_weights(num_experts, hidden, intermediate, wfmt, act, flags=0):
    """-> (weight plan handle, packed_bytes).  flags: MOE_WFLAG_* bits."""
    d = moe_weight_desc(num_experts, hidden, intermediate, WFMT.get(wfmt, wfmt), ACT.get(act, act), flags)
    h, n = _vp(), _sz()
    _check(_lib.moe_plan_weights(ctypes.byref(d), ctypes.byref(h), ctypes.byref(n)), "moe_plan_weights")
    return h.value, n.value


def moe_prepare_weights(wplan, w13_codes, w13_scales, w13_global, w2_codes, w2_scales, w2_global,
                        packed, stream=None):
    _check(_lib.moe_prepare_weights(wplan, _ptr(w13_codes), _ptr(w13_scales), _ptr(w13_global),
                                    _ptr(w2_codes), _ptr(w2_scales), _ptr(w2_global), _ptr(packed),
                                    _stream(stream)), "moe_prepare_weights")


def _caps(wplan, top_k, max_tokens, afmt):
    return moe_caps(wplan, top_k, max_tokens, AFMT.get(afmt, afmt))


def moe_is_supported(wplan, top_k, max_tokens, afmt) -> int:
    """Status code (not raised): MOE_OK when supported."""
    c = _caps(wplan, top_k, max_tokens, afmt)
    return _lib.moe_is_supported(ctypes.byref(c))


def moe_plan(wplan, top_k, max_tokens, afmt):
    """-> (plan handle, scratch_bytes, m_tile)."""
    c = _caps(wplan, top_k, max_tokens, afmt)
    h, n, m = _vp(), _sz(), _i32()
    _check(_lib.moe_plan(ctypes.byref(c), ctypes.byref(h), ctypes.byref(n), ctypes.byref(m)), "moe_plan")
    return h.value, n.value, m.value


def moe_bind(plan, scratch, scratch_bytes, packed, x, topk_ids, topk_weights, num_tokens, out):
    h = _vp()
    _check(_lib.moe_bind(plan, _ptr(scratch), scratch_bytes, _ptr(packed), _ptr(x), _ptr(topk_ids),
                         _ptr(topk_weights), num_tokens, _ptr(out), ctypes.byref(h)), "moe_bind")
    return h.value


def moe_run(binding, stream=None):
    _check(_lib.moe_run(binding, _stream(stream)), "moe_run")


def moe_run_timed(binding, events, stream=None):
    """``events``: MOE_NUM_STAGES+1 raw cudaEvent_t handles (ints) created with timing enabled."""
    arr = (_vp * (MOE_NUM_STAGES + 1))(*events)
    _check(_lib.moe_run_timed(binding, _stream(stream), arr), "moe_run_timed")


MOE_PEAK_F16, MOE_PEAK_FP4, MOE_PEAK_MXFP8 = 0, 1, 2


def moe_measure_mma_peak(kind, n, iters=20000):
    """Back-to-back tcgen05.mma issue rate (TFLOP/s) for kind MOE_PEAK_F16 / MOE_PEAK_FP4 / MOE_PEAK_MXFP8."""
    t = ctypes.c_float(0)
    _check(_lib.moe_measure_mma_peak(kind, n, iters, ctypes.byref(t)), "moe_measure_mma_peak")
    return t.value


def moe_launch_count(binding):
    """Kernels enqueued by the last forward on ``binding``."""
    n = ctypes.c_int32(0)
    _check(_lib.moe_launch_count(binding, ctypes.byref(n)), "moe_launch_count")
    return n.value


def moe_run_host(binding, x_host, ids_host, weights_host, out_host, stream=None):
    _check(_lib.moe_run_host(binding, _ptr(x_host), _ptr(ids_host), _ptr(weights_host), _ptr(out_host),
                             _stream(stream)), "moe_run_host")


def moe_device_status(binding, stream=None):
    """-> (status code, [flags, dropped, 0, 0]); MOE_ERR_TIMEOUT is returned, not raised."""
    st = (_i32 * 4)()
    rc = _lib.moe_device_status(binding, _stream(stream), st)
    if rc not in (MOE_OK, MOE_ERR_TIMEOUT):
        _check(rc, "moe_device_status")
    return rc, list(st)


def moe_debug_hidden(binding, intermediate, rows_cap, stream=None):
    """GEMM1's h of the last run, [rows, I] float32 in sorted-slot order."""
    h = np.zeros((rows_cap, intermediate), np.float32)
    n = _i32()
    _check(_lib.moe_debug_hidden(binding, _stream(stream), h.ctypes.data_as(_P(ctypes.c_float)), rows_cap,
                                 ctypes.byref(n)), "moe_debug_hidden")
    return h[:n.value]


def moe_selftest_wait_timeout(status_dev, stream=None):
    """Let one bounded device wait run out: -> (status code, [flags, 0, 0, 0]).
    MOE_ERR_TIMEOUT is the expected code and is returned, not raised."""
    st = (_i32 * 4)()
    rc = _lib.moe_selftest_wait_timeout(_stream(stream), _ptr(status_dev), st)
    if rc not in (MOE_OK, MOE_ERR_TIMEOUT):
        _check(rc, "moe_selftest_wait_timeout")
    return rc, list(st)


def moe_debug_routing(binding, num_experts, num_pairs, sorted_cap, stream=None):
    counts = np.zeros(num_experts, np.int32)
    offsets = np.zeros(num_experts + 1, np.int32)
    pair_pos = np.zeros(max(num_pairs, 1), np.int32)
    sorted_pair = np.zeros(max(sorted_cap, 1), np.int32)
    ip = lambda a: a.ctypes.data_as(_P(_i32))  # noqa: E731
    _check(_lib.moe_debug_routing(binding, _stream(stream), ip(counts), ip(offsets), ip(pair_pos),
                                  ip(sorted_pair), sorted_cap), "moe_debug_routing")
    return dict(counts=counts, offsets=offsets, pair_pos=pair_pos[:num_pairs],
                sorted_pair=sorted_pair[:offsets[-1]])


def moe_quantize(qfmt, gmode, src, batch, rows, cols, codes, scales, global_, stream=None):
    import torch
    bf16 = int(getattr(src, "dtype", None) == torch.bfloat16)
    _check(_lib.moe_quantize(qfmt, gmode, bf16, _ptr(src), batch, rows, cols, _ptr(codes), _ptr(scales),
                             _ptr(global_), _stream(stream)), "moe_quantize")


def moe_destroy_weight_plan(h):
    _lib.moe_destroy_weight_plan(h)


def moe_destroy_plan(h):
    _lib.moe_destroy_plan(h)


def moe_destroy_binding(h):
    _lib.moe_destroy_binding(h)


def moe_run_no_alloc(plan, packed, x, topk_ids, topk_weights, num_tokens, out, stream=None):
    """Forward with the library's own static scratch, for callers that cannot allocate."""
    _check(_lib.moe_run_no_alloc(plan, _ptr(packed), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                 num_tokens, _ptr(out), _stream(stream)), "moe_run_no_alloc")


def moe_no_alloc_device_status(plan, stream=None):
    """Status word of the last moe_run_no_alloc: -> (status code, [flags, dropped, 0, 0]);
    MOE_ERR_TIMEOUT is returned, not raised."""
    st = (_i32 * 4)()
    rc = _lib.moe_no_alloc_device_status(plan, _stream(stream), st)
    if rc not in (MOE_OK, MOE_ERR_TIMEOUT):
        _check(rc, "moe_no_alloc_device_status")
    return rc, list(st)


def moe_plan_set_option(plan, option, value):
    _check(_lib.moe_plan_set_option(plan, option, value), "moe_plan_set_option")


def moe_selftest_grid_barrier_timeout(binding, stream=None):
    """One single-launch forward with a grid-barrier arrival withheld: -> (status code,
    [flags, dropped, 0, 0]); MOE_ERR_TIMEOUT is the expected code and is returned, not raised."""
    st = (_i32 * 4)()
    rc = _lib.moe_selftest_grid_barrier_timeout(binding, _stream(stream), st)
    if rc not in (MOE_OK, MOE_ERR_TIMEOUT):
        _check(rc, "moe_selftest_grid_barrier_timeout")
    return rc, list(st)
