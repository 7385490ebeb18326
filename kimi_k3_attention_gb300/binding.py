"""Thin ctypes binding of libattnres.so (include/attnres.h).

Argument marshalling only: every step of the op runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors used as device buffers; their data
pointers and the current torch stream are handed to the C ABI.  If the shared
library is missing the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattnres.so")

STATUS = {
    0: "ATTNRES_OK", -1: "ATTNRES_ERR_NULL", -2: "ATTNRES_ERR_SHAPE", -3: "ATTNRES_ERR_ALIGN",
    -4: "ATTNRES_ERR_ALIAS", -5: "ATTNRES_ERR_EPS", -6: "ATTNRES_ERR_CUDA",
    -7: "ATTNRES_ERR_DEVICE", -8: "ATTNRES_ERR_CONFIG", -9: "ATTNRES_ERR_DTYPE",
}
DTYPE_BF16, DTYPE_FP16 = 0, 1
ATTNRES_DEVICE_WAIT_TIMEOUT = 1
VARIANTS = {"auto": 0, "cta": 1, "cluster": 2, "stream": 3, "pipe": 4, "cluster2": 5}

# Every symbol include/attnres.h declares.
EXPORTS = (
    "attnres_add_rmsnorm",
    "attnres_add_rmsnorm_ex",
    "attnres_add_rmsnorm_tap",
    "attnres_add_rmsnorm_f16",
    "attnres_rmsnorm",
    "attnres_tail_add",
    "attnres_tail_add_f16",
    "attnres_access_pattern",
    "attnres_launch",
    "attnres_plan",
    "attnres_plan_host",
    "attnres_status_string",
    "attnres_last_cuda_error",
    "attnres_device_status",
    "attnres_debug_exchange",
    "attnres_version",
)


class AttnResError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("cluster", ctypes.c_int),
                ("threads", ctypes.c_int), ("grid_tokens", ctypes.c_int), ("pdl", ctypes.c_int),
                ("stages", ctypes.c_int), ("prefetch", ctypes.c_int),
                ("tail_tokens", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class Args(ctypes.Structure):
    _fields_ = [("prefix", ctypes.c_void_p), ("add", ctypes.c_void_p), ("add2", ctypes.c_void_p),
                ("bank", ctypes.c_void_p), ("w", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("out", ctypes.c_void_p), ("new_prefix", ctypes.c_void_p),
                ("h_out", ctypes.c_void_p), ("M", ctypes.c_int), ("N", ctypes.c_int),
                ("H", ctypes.c_int), ("fold", ctypes.c_int), ("dtype", ctypes.c_int)]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the shared library once; raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} not found: build it with kimi_k3_attention_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    args = [vp, vp, vp, vp, vp, vp, f, vp, vp, i, i, i, vp]
    lib.attnres_add_rmsnorm.argtypes = args
    lib.attnres_add_rmsnorm.restype = i
    lib.attnres_add_rmsnorm_f16.argtypes = args
    lib.attnres_add_rmsnorm_f16.restype = i
    lib.attnres_add_rmsnorm_ex.argtypes = args + [ctypes.POINTER(Config)]
    lib.attnres_add_rmsnorm_ex.restype = i
    lib.attnres_plan.argtypes = [i, i, i, i, ctypes.POINTER(Config)]
    lib.attnres_plan.restype = i
    lib.attnres_plan_host.argtypes = [i, i, i, i, ctypes.POINTER(Config)]
    lib.attnres_plan_host.restype = i
    lib.attnres_status_string.argtypes = [i]
    lib.attnres_status_string.restype = ctypes.c_char_p
    lib.attnres_last_cuda_error.argtypes = []
    lib.attnres_last_cuda_error.restype = i
    lib.attnres_version.argtypes = []
    lib.attnres_version.restype = i
    lib.attnres_add_rmsnorm_tap.argtypes = [vp, vp, vp, vp, vp, vp, f, vp, vp, vp, i, i, i, vp]
    lib.attnres_add_rmsnorm_tap.restype = i
    lib.attnres_rmsnorm.argtypes = [vp, vp, vp, vp, f, vp, i, i, i, vp]
    lib.attnres_rmsnorm.restype = i
    lib.attnres_tail_add.argtypes = [vp, vp, vp, vp, i, i, vp]
    lib.attnres_tail_add.restype = i
    lib.attnres_tail_add_f16.argtypes = [vp, vp, vp, vp, i, i, vp]
    lib.attnres_tail_add_f16.restype = i
    lib.attnres_access_pattern.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, vp]
    lib.attnres_access_pattern.restype = i
    lib.attnres_launch.argtypes = [ctypes.POINTER(Args), ctypes.POINTER(Config), vp]
    lib.attnres_launch.restype = i
    lib.attnres_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i]
    lib.attnres_device_status.restype = i
    lib.attnres_debug_exchange.argtypes = [i, ctypes.c_longlong]
    lib.attnres_debug_exchange.restype = i
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().attnres_status_string(int(status)).decode()


def _check(status: int):
    if status != 0:
        lib = load()
        msg = lib.attnres_status_string(status).decode()
        if status == -6:
            msg += f" (cudaError {lib.attnres_last_cuda_error()})"
        raise AttnResError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_config(variant="auto", cluster=0, threads=0, grid_tokens=0, pdl=0, stages=0,
                prefetch=0, tail_tokens=0) -> Config:
    v = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    return Config(v, int(cluster), int(threads), int(grid_tokens), int(pdl), int(stages),
                  int(prefetch), int(tail_tokens))


def _dtype_code(t) -> int:
    """ATTNRES_DTYPE_* of a torch tensor (bfloat16 or float16)."""
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float16:
        return DTYPE_FP16
    raise TypeError(f"tensors must be bfloat16 or float16, got {t.dtype}")


def _check_tensor(name, t, shape=None, dtype=None):
    """dtype: the torch dtype every tensor of the call must have (default
    bfloat16)."""
    import torch
    want = torch.bfloat16 if dtype is None else dtype
    if t.dtype != want:
        raise TypeError(f"{name} must be {want}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def attnres_add_rmsnorm(prefix, add, add2, bank, w, gamma, eps, out, new_prefix,
                        stream=None, config: Optional[Config] = None, check=True):
    """Launch the fused epilogue on torch CUDA tensors (see include/attnres.h).

    prefix, add, add2 (or None), out, new_prefix: [M, H]; bank: [N, M, H];
    w, gamma: [H]; all bfloat16 (or all float16), contiguous, on the current
    device.
    stream: a torch.cuda.Stream (default: the current stream).
    config: a Config pinning the launch (default: the library's choice).
    """
    N, M, H = bank.shape
    dt = prefix.dtype
    if check:
        _dtype_code(prefix)
        for name, t, shp in (("prefix", prefix, (M, H)), ("add", add, (M, H)),
                             ("bank", bank, (N, M, H)), ("w", w, (H,)), ("gamma", gamma, (H,)),
                             ("out", out, (M, H)), ("new_prefix", new_prefix, (M, H))):
            _check_tensor(name, t, shp, dt)
        if add2 is not None:
            _check_tensor("add2", add2, (M, H), dt)
    lib = load()
    s = _stream_handle(stream)
    if _dtype_code(prefix) == DTYPE_FP16:
        if config is None:
            st = lib.attnres_add_rmsnorm_f16(_ptr(prefix), _ptr(add), _ptr(add2), _ptr(bank),
                                             _ptr(w), _ptr(gamma), float(eps), _ptr(out),
                                             _ptr(new_prefix), M, N, H, s)
            _check(st)
        else:
            launch(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, config=config,
                   stream=stream)
        return
    if config is None:
        st = lib.attnres_add_rmsnorm(_ptr(prefix), _ptr(add), _ptr(add2), _ptr(bank), _ptr(w),
                                     _ptr(gamma), float(eps), _ptr(out), _ptr(new_prefix),
                                     M, N, H, s)
    else:
        st = lib.attnres_add_rmsnorm_ex(_ptr(prefix), _ptr(add), _ptr(add2), _ptr(bank), _ptr(w),
                                        _ptr(gamma), float(eps), _ptr(out), _ptr(new_prefix),
                                        M, N, H, s, ctypes.byref(config))
    _check(st)


def attnres_add_rmsnorm_tap(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, h_out,
                            stream=None):
    """The fused epilogue that also writes h_out = bf16(h), the pre-norm mixture
    (fp16(h) for float16 tensors)."""
    N, M, H = bank.shape
    _check_tensor("h_out", h_out, (M, H), prefix.dtype)
    if _dtype_code(prefix) == DTYPE_FP16:
        launch(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, h_out=h_out, stream=stream)
        return
    _check(load().attnres_add_rmsnorm_tap(_ptr(prefix), _ptr(add), _ptr(add2), _ptr(bank),
                                          _ptr(w), _ptr(gamma), float(eps), _ptr(out),
                                          _ptr(new_prefix), _ptr(h_out), M, N, H,
                                          _stream_handle(stream)))


def attnres_rmsnorm(prefix, bank, w, gamma, eps, out, stream=None, config: Optional[Config] = None):
    """The attention-residual + RMSNorm alone: sources bank[0..N-1] and prefix."""
    N, M, H = bank.shape
    _dtype_code(prefix)
    for name, t, shp in (("prefix", prefix, (M, H)), ("bank", bank, (N, M, H)), ("w", w, (H,)),
                         ("gamma", gamma, (H,)), ("out", out, (M, H))):
        _check_tensor(name, t, shp, prefix.dtype)
    if config is None and _dtype_code(prefix) == DTYPE_BF16:
        _check(load().attnres_rmsnorm(_ptr(prefix), _ptr(bank), _ptr(w), _ptr(gamma), float(eps),
                                      _ptr(out), M, N, H, _stream_handle(stream)))
    else:
        launch(prefix, None, None, bank, w, gamma, eps, out, None, M=M, N=N, H=H, fold=False,
               config=config, stream=stream)


def attnres_tail_add(prefix, add, add2, new_prefix, stream=None):
    """The standalone fold: new_prefix = bf16(prefix + bf16(add + add2))
    (fp16(prefix + fp16(add + add2)) for float16 tensors)."""
    M, H = prefix.shape
    dt = prefix.dtype
    code = _dtype_code(prefix)
    for name, t in (("prefix", prefix), ("add", add), ("new_prefix", new_prefix)):
        _check_tensor(name, t, (M, H), dt)
    if add2 is not None:
        _check_tensor("add2", add2, (M, H), dt)
    lib = load()
    fn = lib.attnres_tail_add_f16 if code == DTYPE_FP16 else lib.attnres_tail_add
    _check(fn(_ptr(prefix), _ptr(add), _ptr(add2), _ptr(new_prefix), M, H, _stream_handle(stream)))


def attnres_access_pattern(prefix, add, add2, bank, out, new_prefix, stream=None):
    """The fused op's memory traffic without its arithmetic (a measurement
    aid): new_prefix = prefix, out = XOR of the N+3 input rows."""
    N, M, H = bank.shape
    dt = prefix.dtype
    for name, t, shp in (("prefix", prefix, (M, H)), ("add", add, (M, H)), ("add2", add2, (M, H)),
                         ("bank", bank, (N, M, H)), ("out", out, (M, H)),
                         ("new_prefix", new_prefix, (M, H))):
        _check_tensor(name, t, shp, dt)
    _check(load().attnres_access_pattern(_ptr(prefix), _ptr(add), _ptr(add2), _ptr(bank), _ptr(out),
                                         _ptr(new_prefix), M, N, H, _stream_handle(stream)))


def launch(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, h_out=None, M=None, N=None,
           H=None, fold=True, config: Optional[Config] = None, stream=None, dtype=None):
    """attnres_launch: any fused call with an optional pinned configuration.
    dtype: DTYPE_BF16 or DTYPE_FP16 (default: that of `prefix`)."""
    if M is None:
        N, M, H = bank.shape
    if dtype is None:
        dtype = _dtype_code(prefix)
    a = Args(_ptr(prefix), _ptr(add), _ptr(add2), _ptr(bank), _ptr(w), _ptr(gamma), float(eps),
             _ptr(out), _ptr(new_prefix), _ptr(h_out), int(M), int(N), int(H), int(bool(fold)),
             int(dtype))
    _check(load().attnres_launch(ctypes.byref(a), None if config is None else ctypes.byref(config),
                                 _stream_handle(stream)))


def attnres_add_rmsnorm_raw(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, M, N, H,
                            stream=0, config: Optional[Config] = None) -> int:
    """The C entry point on raw integer pointers; returns the status code."""
    lib = load()
    vp = ctypes.c_void_p
    args = [vp(prefix), vp(add), vp(add2) if add2 else None, vp(bank), vp(w), vp(gamma),
            float(eps), vp(out), vp(new_prefix), int(M), int(N), int(H), vp(stream)]
    if config is None:
        return lib.attnres_add_rmsnorm(*args)
    return lib.attnres_add_rmsnorm_ex(*args, ctypes.byref(config))


def attnres_plan(M, N, H, has_add2=True) -> dict:
    c = Config()
    _check(load().attnres_plan(int(M), int(N), int(H), int(bool(has_add2)), ctypes.byref(c)))
    return c.as_dict()


def attnres_plan_host(M, N, H, has_add2=True) -> dict:
    """The automatic launch configuration, computed without a CUDA device."""
    c = Config()
    _check(load().attnres_plan_host(int(M), int(N), int(H), int(bool(has_add2)), ctypes.byref(c)))
    return c.as_dict()


def version() -> int:
    return load().attnres_version()


def device_status(clear=False) -> int:
    """The kernels' status bits on the current device (0 = no failure)."""
    v = ctypes.c_uint(0)
    _check(load().attnres_device_status(ctypes.byref(v), int(bool(clear))))
    return v.value


def debug_exchange(extra_bytes=0, wait_ns=0):
    """Test hook: make every exchange wait for bytes that never come."""
    _check(load().attnres_debug_exchange(int(extra_bytes), int(wait_ns)))
