"""The kernels' failure path on the GPU, without a fault: a test hook makes
every exchange of partial sums wait for bytes that never come; the waits
must expire, the kernel must finish and report it in the library's status
word, and normal calls must work again afterwards."""
import pytest
import torch

from kimi_k3_attention_gb300 import binding
from kimi_k3_attention_gb300 import workloads as wl

from oracle import fold

from gpu_helpers import assert_parity, fmt_of, run_gpu, u16

pytestmark = pytest.mark.gpu

H = wl.H_MODEL


@pytest.fixture(autouse=True)
def _restore():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.device_status(clear=True)
    yield
    binding.debug_exchange(0, 0)
    binding.device_status(clear=True)


@pytest.mark.parametrize("cfg,N,dtype", [
    (binding.make_config("cluster", cluster=4), 3, torch.bfloat16),
    (binding.make_config("cluster", cluster=16), 3, torch.bfloat16),
    (binding.make_config("pipe", cluster=4, grid_tokens=2), 3, torch.bfloat16),
    (binding.make_config("cta"), 3, torch.bfloat16),
    (binding.make_config("cluster", cluster=8), 20, torch.bfloat16),
    (binding.make_config("stream", cluster=7, grid_tokens=2), 31, torch.bfloat16),
    (binding.make_config("stream", cluster=7, grid_tokens=2), 12, torch.float16),
], ids=["cluster4", "cluster16", "pipe4", "cta", "deep-cluster8", "deep-stream7-walk",
        "fp16-stream7-walk"])
def test_exchange_wait_expires_and_reports(cfg, N, dtype):
    inp = wl.make_inputs(5, N, H, seed=81, dtype=dtype).to("cuda")
    out = torch.empty_like(inp.prefix)
    newp = torch.empty_like(inp.prefix)
    binding.debug_exchange(extra_bytes=4, wait_ns=2_000_000)      # 2 ms
    binding.attnres_add_rmsnorm(inp.prefix, inp.add, inp.add2, inp.bank, inp.w, inp.gamma,
                                inp.eps, out, newp, config=cfg)
    torch.cuda.synchronize()                                        # finishes, no hang
    status = binding.device_status(clear=True)
    assert status & binding.ATTNRES_DEVICE_WAIT_TIMEOUT
    # outputs built from partial sums are marked, not passed off as results;
    # the fold does not depend on the exchange
    assert torch.isnan(out.float()).all()
    ref_np, _ = fold(u16(inp.prefix), u16(inp.add), u16(inp.add2), fmt_of(inp))
    assert (u16(newp) == ref_np).all()
    binding.debug_exchange(0, 0)
    gnp, gout = run_gpu(inp.to("cpu"), cfg)                         # normal again
    assert_parity(inp.to("cpu"), gnp, gout)


def test_debug_hook_bounds():
    with pytest.raises(binding.AttnResError):
        binding.debug_exchange(extra_bytes=-1)
    with pytest.raises(binding.AttnResError):
        binding.debug_exchange(extra_bytes=4, wait_ns=11 * 10 ** 9)
