"""ctypes binding of libfa.so (include/fa.h), argument marshalling only.

Every function named ``fa_*`` here has the name and argument order of the C
entry point and passes torch tensors' device pointers plus the current torch
stream.  All arithmetic runs in the CUDA kernels of libfa.so; nothing here
computes attention.  If libfa.so is missing or fails to load, every call
raises FaError: there is no fallback.
"""

from __future__ import annotations

import ctypes
import math
import os
import re
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "fa.h")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_NO_MEMORY = 4
FA_ERR_TIMEOUT = 5
FA_ERR_SCRATCH_TOO_SMALL = 6
FA_BWD_NOALLOC_SCRATCH_BYTES = 64 << 20
FA_CAUSAL_NONE = 0
FA_CAUSAL_TOP_LEFT = 1
FA_CAUSAL_BOTTOM_RIGHT = 2
_CAUSAL_NAMES = {"none": FA_CAUSAL_NONE, "top_left": FA_CAUSAL_TOP_LEFT, "bottom_right": FA_CAUSAL_BOTTOM_RIGHT}


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _strerror(status) if _lib is not None else f"fa_status {status}"
        super().__init__(f"{what}: {msg}" if what else msg)


_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_u64 = ctypes.c_uint64

_SIGNATURES = {
    "fa_fwd": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_fwd_ex": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_fwd_gqa": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_bwd_gqa": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_bwd_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_fwd_general": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_bwd_general": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_poll_status": ([_vp], _i),
    "fa_set_wait_timeout_ns": ([_u64], _u64),
    "fa_selftest_wait_timeout": ([_u64, _vp], _i),
    "fa_strerror": ([_i], ctypes.c_char_p),
    "fa_abi_version": ([], _i),
    "fa_trim_workspace": ([], _i),
    "fa_timing_enable": ([_i], _i),
    "fa_timing_read": ([_i, ctypes.POINTER(_i), ctypes.POINTER(ctypes.c_double)], _i),
    "fa_launch_count": ([_i, ctypes.POINTER(ctypes.c_uint64)], _i),
}


class FwdPlan(ctypes.Structure):
    """fa_fwd_plan_t (include/fa.h)."""
    _fields_ = [(n, _i) for n in ("packed_heads", "unit_heads", "unit_rows", "query_block", "key_tile",
                                  "key_tiles", "num_splits", "key_tiles_per_split", "dual", "partials",
                                  "num_units", "grid", "head_window", "launches")] + [("workspace_bytes", _u64)]


class BwdPlan(ctypes.Structure):
    """fa_bwd_plan_t (include/fa.h)."""
    _fields_ = [(n, _i) for n in ("q_tiles", "k_tiles", "q_tile_first", "kv_tiles_used", "dq_units", "dq_grid",
                                  "kv_units", "kv_cta_pair", "kv_passes", "launches")] + [
        (n, _u64) for n in ("zeroed_dq_bytes", "zeroed_dkdv_bytes", "workspace_bytes")]


_SIGNATURES["fa_fwd_plan"] = ([_i] * 9 + [_u64, ctypes.POINTER(FwdPlan)], _i)
_SIGNATURES["fa_bwd_plan"] = ([_i] * 8 + [ctypes.POINTER(BwdPlan)], _i)


def load():
    """Load libfa.so once; raise FaError if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise FaError(FA_ERR_CUDA, f"{LIB_PATH} is not built (run exact_attention_92_gb300.build.build())")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def declared_symbols():
    """Entry points declared in include/fa.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|uint64_t|const char\*)\s+(fa_\w+)\s*\(", text, re.M)))


def _strerror(status: int) -> str:
    return load().fa_strerror(int(status)).decode()


def _check(status: int, what: str):
    if status != FA_OK:
        raise FaError(status, what)


def _stream_ptr(stream, device):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _check_bhnd(name, t, shape=None):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    # The library works on the current CUDA device (its status word, its
    # scratch and its launches); a tensor on another device would be read
    # through the wrong device's context.
    if t.device.index is not None and t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()} (use torch.cuda.device)")


def _check_lse(t, shape):
    import torch

    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
            and tuple(t.shape) == tuple(shape)):
        raise ValueError(f"lse must be a contiguous float32 CUDA tensor of shape {tuple(shape)}")


def _scale(scale, d):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


# ---------------------------------------------------------------- C names

def fa_fwd(q, k, v, o, lse, causal=False, scale=None, stream=None):
    """C fa_fwd: O and LSE of softmax(scale Q K^T [+ causal mask]) V."""
    return fa_fwd_ex(q, k, v, o, lse, causal, scale, 0, stream)


def fa_fwd_ex(q, k, v, o, lse, causal=False, scale=None, num_splits=0, stream=None):
    """C fa_fwd_ex: fa_fwd with an explicit key-split count (0 = automatic)."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o)):
        _check_bhnd(name, t, q.shape)
    _check_lse(lse, (B, H, N))
    lib = load()
    st = lib.fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, 1 if causal else 0,
                       _scale(scale, d), int(num_splits), _stream_ptr(stream, q.device))
    _check(st, "fa_fwd_ex")


def fa_fwd_gqa(q, k, v, o, lse, causal=False, scale=None, num_splits=0, stream=None):
    """C fa_fwd_gqa: grouped-query attention; q, o [B, H, N, d], k, v
    [B, Hkv, N, d] with Hkv dividing H (query head h reads key/value head
    h // (H // Hkv))."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    _check_bhnd("k", k)
    Hkv = k.shape[1]
    _check_bhnd("k", k, (B, Hkv, N, d))
    _check_bhnd("v", v, (B, Hkv, N, d))
    _check_bhnd("o", o, q.shape)
    _check_lse(lse, (B, H, N))
    lib = load()
    st = lib.fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d, 1 if causal else 0,
                        _scale(scale, d), int(num_splits), _stream_ptr(stream, q.device))
    _check(st, "fa_fwd_gqa")


def _causal_code(causal):
    """False/True (top-left), or a FA_CAUSAL_* code, or its name."""
    if isinstance(causal, str):
        if causal not in _CAUSAL_NAMES:
            raise ValueError(f"causal must be one of {sorted(_CAUSAL_NAMES)}, got {causal!r}")
        return _CAUSAL_NAMES[causal]
    if isinstance(causal, bool):
        return FA_CAUSAL_TOP_LEFT if causal else FA_CAUSAL_NONE
    return int(causal)


def fa_fwd_general(q, k, v, o, lse, causal=False, scale=None, num_splits=0, stream=None):
    """C fa_fwd_general: q, o [B, H, Nq, d], k, v [B, Hkv, Nk, d];
    causal False / True (top-left) / "top_left" / "bottom_right" or a
    FA_CAUSAL_* code."""
    _check_bhnd("q", q)
    B, H, Nq, d = q.shape
    _check_bhnd("k", k)
    Hkv, Nk = k.shape[1], k.shape[2]
    _check_bhnd("k", k, (B, Hkv, Nk, d))
    _check_bhnd("v", v, (B, Hkv, Nk, d))
    _check_bhnd("o", o, q.shape)
    _check_lse(lse, (B, H, Nq))
    lib = load()
    st = lib.fa_fwd_general(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Nq, Nk, d,
                            _causal_code(causal), _scale(scale, d), int(num_splits), _stream_ptr(stream, q.device))
    _check(st, "fa_fwd_general")


def fa_bwd_general(q, k, v, o, lse, dout, dq, dk, dv, causal=False, scale=None, stream=None):
    """C fa_bwd_general: gradients for fa_fwd_general (same shapes and
    causal argument); dk, dv have the shape of k, v."""
    _check_bhnd("q", q)
    B, H, Nq, d = q.shape
    _check_bhnd("k", k)
    Hkv, Nk = k.shape[1], k.shape[2]
    for name, t in (("k", k), ("v", v), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, (B, Hkv, Nk, d))
    for name, t in (("o", o), ("dout", dout), ("dq", dq)):
        _check_bhnd(name, t, q.shape)
    _check_lse(lse, (B, H, Nq))
    lib = load()
    st = lib.fa_bwd_general(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                            _ptr(dv), B, H, Hkv, Nq, Nk, d, _causal_code(causal), _scale(scale, d),
                            _stream_ptr(stream, q.device))
    _check(st, "fa_bwd_general")


def fa_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, causal=False, scale=None, stream=None):
    """C fa_bwd_gqa: gradients for grouped-query attention; dk, dv have the
    shape of k, v ([B, Hkv, N, d]) and hold the sums over each group."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    _check_bhnd("k", k)
    Hkv = k.shape[1]
    for name, t in (("k", k), ("v", v), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, (B, Hkv, N, d))
    for name, t in (("o", o), ("dout", dout), ("dq", dq)):
        _check_bhnd(name, t, q.shape)
    _check_lse(lse, (B, H, N))
    lib = load()
    st = lib.fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, H, Hkv, N, d, 1 if causal else 0, _scale(scale, d), _stream_ptr(stream, q.device))
    _check(st, "fa_bwd_gqa")


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal=False, scale=None, stream=None):
    """C fa_bwd: dQ, dK, dV from the forward inputs, O, LSE and dO."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, q.shape)
    _check_lse(lse, (B, H, N))
    lib = load()
    st = lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                    B, H, N, d, 1 if causal else 0, _scale(scale, d), _stream_ptr(stream, q.device))
    _check(st, "fa_bwd")


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, causal=False, scale=None, stream=None):
    """C fa_bwd_noalloc: fa_bwd with its workspace in the library's static
    device scratch (no device allocation; see include/fa.h)."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, q.shape)
    _check_lse(lse, (B, H, N))
    lib = load()
    st = lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                            _ptr(dv), B, H, N, d, 1 if causal else 0, _scale(scale, d),
                            _stream_ptr(stream, q.device))
    _check(st, "fa_bwd_noalloc")


def fa_poll_status(stream=None):
    """C fa_poll_status: synchronise the stream, return and clear the device status."""
    import torch

    return load().fa_poll_status(_stream_ptr(stream, torch.device("cuda")))


def fa_set_wait_timeout_ns(ns: int) -> int:
    return int(load().fa_set_wait_timeout_ns(int(ns)))


def fa_selftest_wait_timeout(timeout_ns: int, stream=None):
    import torch

    _check(load().fa_selftest_wait_timeout(int(timeout_ns), _stream_ptr(stream, torch.device("cuda"))),
           "fa_selftest_wait_timeout")


def fa_strerror(status: int) -> str:
    return _strerror(status)


def fa_abi_version() -> int:
    return int(load().fa_abi_version())


def fa_trim_workspace() -> None:
    """C fa_trim_workspace: give back the workspace memory the library's pool
    keeps reserved on the current device."""
    _check(load().fa_trim_workspace(), "fa_trim_workspace")


def fa_timing_enable(on: bool) -> None:
    _check(load().fa_timing_enable(1 if on else 0), "fa_timing_enable")


def fa_timing_read(kernel: int):
    """(launches, total milliseconds) of one kernel since timing was enabled or last read."""
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    _check(load().fa_timing_read(int(kernel), ctypes.byref(n), ctypes.byref(ms)), "fa_timing_read")
    return n.value, ms.value


def fa_launch_count(kernel: int) -> int:
    """Launches of one library kernel since the library was loaded."""
    n = ctypes.c_uint64(0)
    _check(load().fa_launch_count(int(kernel), ctypes.byref(n)), "fa_launch_count")
    return n.value


def _plan_dict(plan):
    return {name: getattr(plan, name) for name, _ in plan._fields_}


def fa_fwd_plan(B, H, Hkv, Nq, Nk, d, causal, num_splits, sm_count, l2_bytes):
    """C fa_fwd_plan: the launch plan of fa_fwd_general for these sizes on a
    device with sm_count SMs and l2_bytes of L2, as a dict of the
    fa_fwd_plan_t fields.  Host only; raises FaError on a refused size."""
    plan = FwdPlan()
    _check(load().fa_fwd_plan(int(B), int(H), int(Hkv), int(Nq), int(Nk), int(d), _causal_code(causal),
                              int(num_splits), int(sm_count), int(l2_bytes), ctypes.byref(plan)), "fa_fwd_plan")
    return _plan_dict(plan)


def fa_bwd_plan(B, H, Hkv, Nq, Nk, d, causal, sm_count):
    """C fa_bwd_plan: the launch plan of fa_bwd_general, as a dict of the
    fa_bwd_plan_t fields.  Host only; raises FaError on a refused size."""
    plan = BwdPlan()
    _check(load().fa_bwd_plan(int(B), int(H), int(Hkv), int(Nq), int(Nk), int(d), _causal_code(causal),
                              int(sm_count), ctypes.byref(plan)), "fa_bwd_plan")
    return _plan_dict(plan)


# ------------------------------------------------------- convenience calls

def forward(q, k, v, causal=False, scale=None, num_splits=0):
    """Allocate O and LSE and run the forward pass; returns (o, lse).  k, v
    may have fewer heads (grouped-query) or another length than q
    (fa_fwd_general; causal may then be "top_left" or "bottom_right")."""
    import torch

    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if tuple(k.shape) == tuple(q.shape) and not isinstance(causal, str):
        fa_fwd_ex(q, k, v, o, lse, causal, scale, num_splits)
    else:
        fa_fwd_general(q, k, v, o, lse, causal, scale, num_splits)
    return o, lse


def backward(q, k, v, o, lse, dout, causal=False, scale=None):
    """Allocate dQ, dK, dV and run the backward pass; returns (dq, dk, dv)
    (shapes and causal argument as for ``forward``)."""
    import torch

    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    if tuple(k.shape) == tuple(q.shape) and not isinstance(causal, str):
        fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal, scale)
    else:
        fa_bwd_general(q, k, v, o, lse, dout, dq, dk, dv, causal, scale)
    return dq, dk, dv
