"""GB300-native fused AttnRes + add2 + RMSNorm decode epilogue.

The op lives in libattnres.so (C ABI in include/attnres.h, CUDA kernels for
sm_103a in csrc/); `binding` is a thin ctypes layer over it.  Build with
`kimi_k3_attention_gb300.build.build()`.
"""
from .binding import (  # noqa: F401
    AttnResError,
    Config,
    attnres_add_rmsnorm,
    attnres_add_rmsnorm_raw,
    attnres_add_rmsnorm_tap,
    attnres_plan,
    attnres_rmsnorm,
    attnres_tail_add,
    launch,
    make_config,
)
