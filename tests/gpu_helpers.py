"""Shared plumbing of the GPU parity tests: device copies of seeded inputs,
guarded output buffers, the C-ABI call, and the comparison with the oracle."""
import numpy as np
import torch

from kimi_k3_attention_gb300 import binding
from oracle import attnres_add_rmsnorm as oracle_op
from oracle import check_out

GUARD = 4096          # BF16 elements of canary on each side of an output
CANARY = 0x5A5A      # a finite BF16 value no correct call writes by chance


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


class Guarded:
    """A [M, H] BF16 (or FP16) device tensor with canary bands before and
    after it."""

    def __init__(self, shape, device="cuda", dtype=torch.bfloat16):
        n = int(np.prod(shape))
        self.buf = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.int16, device=device)
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(*shape)

    def guards_intact(self) -> bool:
        b = self.buf.cpu()
        return bool((b[:GUARD] == CANARY).all() and (b[-GUARD:] == CANARY).all())


def run_gpu(inp, config=None, stream=None):
    """Run the op through the C ABI on device copies of `inp` (an Inputs on
    the CPU or the GPU).  Returns (new_prefix_bits, out_bits) as numpy."""
    d = inp.to("cuda")
    out = Guarded((inp.M, inp.H), dtype=inp.prefix.dtype)
    newp = Guarded((inp.M, inp.H), dtype=inp.prefix.dtype)
    binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps,
                                out.t, newp.t, stream=stream, config=config)
    torch.cuda.synchronize()
    assert binding.device_status() == 0, "a kernel reported a failure"
    assert out.guards_intact(), "write outside out"
    assert newp.guards_intact(), "write outside new_prefix"
    return u16(newp.t), u16(out.t)


def fmt_of(inp) -> str:
    """The oracle's name of the element format of an Inputs."""
    return "fp16" if inp.prefix.dtype == torch.float16 else "bf16"


def oracle(inp, tokens=None):
    return oracle_op(u16(inp.prefix), u16(inp.add), None if inp.add2 is None else u16(inp.add2),
                     u16(inp.bank), u16(inp.w), u16(inp.gamma), inp.eps, tokens=tokens,
                     fmt=fmt_of(inp))


def assert_parity(inp, gpu_np, gpu_out, tokens=None, label=""):
    ref_np, ref_out, bound = oracle(inp, tokens)
    if tokens is not None:
        gpu_np, gpu_out = gpu_np[tokens], gpu_out[tokens]
    bad = np.flatnonzero((gpu_np != ref_np).ravel())
    assert bad.size == 0, (f"{label}: new_prefix differs at {bad.size} elements, first flat index "
                           f"{bad[0]}: gpu {gpu_np.ravel()[bad[0]]:#06x} oracle {ref_np.ravel()[bad[0]]:#06x}")
    r = check_out(gpu_out, ref_out, bound, fmt_of(inp))
    assert r["ok"], f"{label}: out outside tolerance: {r}"
    return r


def _ceil(a, b):
    return -(-a // b)


def split_configs(H):
    """Every cluster size whose CTAs fit the split shape (<= 256 threads of 8
    columns; registers uncapped, or capped for two CTAs per SM), the
    register-capped streaming shape (<= 224 threads) or the pipelined
    persistent kernel (<= 256 threads) for this H, the one-CTA-per-token
    variant where it fits (<= 448 threads of 16 columns), and the automatic
    choice (None)."""
    H8 = H // 8
    cfgs = [None]
    for c in range(1, 17):
        if _ceil(_ceil(H8, c), 32) * 32 <= 256:
            cfgs.append(binding.make_config("cluster", cluster=c))
    for c in range(1, 17):
        if _ceil(_ceil(H8, c), 32) * 32 <= 256:
            cfgs.append(binding.make_config("cluster2", cluster=c))
    for c in range(1, 17):
        if _ceil(_ceil(H8, c), 32) * 32 <= 224:
            cfgs.append(binding.make_config("stream", cluster=c))
    for c in range(1, 17):
        if _ceil(_ceil(H8, c), 32) * 32 <= 256:
            cfgs.append(binding.make_config("pipe", cluster=c))
    if _ceil(_ceil(H8, 2), 32) * 32 <= 448:
        cfgs.append(binding.make_config("cta"))
    return cfgs


def cfg_name(c):
    if c is None:
        return "auto"
    d = c.as_dict()
    if d["variant"] == 1:
        return "cta"
    name = {2: "cluster", 3: "stream", 4: "pipe", 5: "cluster2"}[d["variant"]]
    extra = f"s{d['stages']}" if d["stages"] else ""
    return f"{name}{d['cluster']}{extra}"
