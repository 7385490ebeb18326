"""CPU oracle for the fused AttnRes + add2 + RMSNorm epilogue.

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by
the CPU-baseline leg of bench.py.  The CUDA library never imports it and it
imports nothing from the library.
"""
from .attnres_oracle import (  # noqa: F401
    algorithmic_bytes,
    attnres_add_rmsnorm,
    attnres_rmsnorm,
    bf16_decode,
    bf16_encode_rne,
    fold,
    mixture,
)
from .tolerance import check_out, ulp_bf16  # noqa: F401
