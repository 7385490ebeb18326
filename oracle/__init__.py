"""CPU oracle for the fused AttnRes + add2 + RMSNorm epilogue.

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by
the CPU-baseline leg of bench.py.  The CUDA library never imports it and it
imports nothing from the library.
"""
from .attnres_oracle import (  # noqa: F401
    BF16,
    FP16,
    Format,
    algorithmic_bytes,
    attnres_add_rmsnorm,
    attnres_rmsnorm,
    bf16_decode,
    bf16_encode_rne,
    decode,
    encode_rne,
    fold,
    fp16_decode,
    fp16_encode_rne,
    mixture,
)
from .tolerance import check_out, ulp, ulp_bf16  # noqa: F401
