"""GPU parity of deep banks, 13 <= N <= 31 snapshots, through the C ABI.

TensorRT-LLM PR #20546 (section "Op") leaves the fused path for N > 12; this
library fuses those too, in the split shape and a register-capped streaming
shape of their own, with the per-token sums reduced in two warp-wide groups
once there are more than 16 sources.  The cases below
cover both sides of that boundary (N = 15 fills one group, 16 starts the
second, 31 fills both), every cluster size, ragged widths, clusters that walk
several tokens, the call without add2, the attention-residual alone with the
tap, and the launch shapes that are not compiled for deep banks."""
import numpy as np
import pytest
import torch

from kimi_k3_attention_gb300 import binding
from kimi_k3_attention_gb300 import workloads as wl
from oracle import attnres_add_rmsnorm as oracle_op
from oracle import attnres_rmsnorm as oracle_alone
from oracle import bf16_decode, check_out

from gpu_helpers import Guarded, assert_parity, cfg_name, run_gpu, u16

pytestmark = pytest.mark.gpu

H = wl.H_MODEL


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def _ceil(a, b):
    return -(-a // b)


def deep_configs(H):
    """The automatic choice, every cluster size of the split shape (<= 256
    threads of 8 columns) and of the deep streaming shape (<= 128 threads)
    that fits this H."""
    need = [_ceil(_ceil(H // 8, c), 32) * 32 for c in range(17)[1:]]
    return ([None] + [binding.make_config("cluster", cluster=c) for c, t in enumerate(need, 1) if t <= 256]
            + [binding.make_config("stream", cluster=c) for c, t in enumerate(need, 1) if t <= 128])


@pytest.mark.parametrize("N", [13, 15, 16, 17, 24, 31])
@pytest.mark.parametrize("M", [1, 8, 32, 64, 300])
@pytest.mark.parametrize("add2", [True, False])
def test_deep_parity_auto(M, N, add2):
    inp = wl.make_inputs(M, N, H, seed=5000 + 64 * M + N, add2=add2)
    np_, out = run_gpu(inp)
    assert_parity(inp, np_, out, label=f"M={M} N={N} add2={add2}")


@pytest.mark.parametrize("N", [13, 16, 22, 23, 31])
def test_deep_every_cluster_size(N):
    inp = wl.make_inputs(5, N, H, seed=5100 + N)
    ref = None
    for cfg in deep_configs(H):
        np_, out = run_gpu(inp, config=cfg)
        assert_parity(inp, np_, out, label=f"N={N} {cfg_name(cfg)}")
        if ref is None:
            ref = np_
        assert (np_ == ref).all()


@pytest.mark.parametrize("Hr,N", [(8, 31), (1000, 17), (1000, 31), (7176, 20), (16384, 31)])
def test_deep_ragged_width(Hr, N):
    inp = wl.make_inputs(3, N, Hr, seed=5200 + Hr + N)
    for cfg in deep_configs(Hr):
        np_, out = run_gpu(inp, config=cfg)
        assert_parity(inp, np_, out, label=f"H={Hr} N={N} {cfg_name(cfg)}")


@pytest.mark.parametrize("N", [14, 31])
@pytest.mark.parametrize("grid,prefetch", [(3, 0), (3, -1), (3, 4), (7, 5), (1, 0)])
def test_deep_walking_clusters(N, grid, prefetch):
    """A few clusters walk all tokens (with and without the next-token L2
    prefetch); the last token of each walk has no successor to prefetch."""
    inp = wl.make_inputs(50, N, H, seed=5300 + N + grid)
    for v in ("cluster", "stream"):
        cfg = binding.make_config(v, cluster=7, grid_tokens=grid, prefetch=prefetch)
        np_, out = run_gpu(inp, config=cfg)
        assert_parity(inp, np_, out, label=f"N={N} {v} grid={grid} prefetch={prefetch}")


@pytest.mark.parametrize("k", [0, 15, 16, 24, 31])
def test_deep_dominant_source(k):
    """w points along source k (source 31 is the updated prefix): alpha is
    close to e_k, so a source sum taken from the wrong group or lane would
    pick another row and miss by far more than the tolerance."""
    N, M = 31, 4
    inp = wl.make_inputs(M, N, H, seed=5400 + k)
    ref_np = oracle_op(u16(inp.prefix), u16(inp.add), u16(inp.add2), u16(inp.bank), u16(inp.w),
                       u16(inp.gamma), inp.eps)[0]
    src = u16(inp.bank)[k, 0] if k < N else ref_np[0]
    w = torch.from_numpy(bf16_decode(src).astype(np.float32) * 0.05).to(torch.bfloat16)
    inp = wl.Inputs(inp.prefix, inp.add, inp.add2, inp.bank, w, inp.gamma, inp.eps)
    np_, out = run_gpu(inp)
    assert_parity(inp, np_, out, label=f"k={k}")


def test_deep_deterministic_and_add2_equals_presummed():
    N, M = 27, 16
    inp = wl.make_inputs(M, N, H, seed=5500)
    a = run_gpu(inp)
    b = run_gpu(inp)
    assert (a[0] == b[0]).all() and (a[1] == b[1]).all()
    s = (inp.add.float() + inp.add2.float()).to(torch.bfloat16)
    pre = wl.Inputs(inp.prefix, s, None, inp.bank, inp.w, inp.gamma, inp.eps)
    c = run_gpu(pre)
    assert (a[0] == c[0]).all() and (a[1] == c[1]).all()


@pytest.mark.parametrize("M,N", [(1, 13), (32, 20), (200, 31)])
def test_deep_alone_and_tap(M, N):
    inp = wl.make_inputs(M, N, H, seed=5600 + M + N)
    d = inp.to("cuda")
    out, hout = Guarded((M, H)), Guarded((M, H))
    binding.launch(d.prefix, None, None, d.bank, d.w, d.gamma, d.eps, out.t, None, h_out=hout.t,
                   fold=False)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert out.guards_intact() and hout.guards_intact()
    ref_out, bound, h, hb = oracle_alone(u16(inp.prefix), u16(inp.bank), u16(inp.w),
                                         u16(inp.gamma), inp.eps, with_h=True)
    r = check_out(u16(out.t), ref_out, bound)
    assert r["ok"], r
    r = check_out(u16(hout.t), h, hb)
    assert r["ok"], r

    out2, newp, hout2 = Guarded((M, H)), Guarded((M, H)), Guarded((M, H))
    binding.attnres_add_rmsnorm_tap(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps,
                                    out2.t, newp.t, hout2.t)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert out2.guards_intact() and newp.guards_intact() and hout2.guards_intact()
    ref_np, ref_out, bound, h, hb = oracle_op(u16(inp.prefix), u16(inp.add), u16(inp.add2),
                                              u16(inp.bank), u16(inp.w), u16(inp.gamma), inp.eps,
                                              with_h=True)
    assert (u16(newp.t) == ref_np).all()
    assert check_out(u16(out2.t), ref_out, bound)["ok"]
    assert check_out(u16(hout2.t), h, hb)["ok"]


@pytest.mark.parametrize("cfg", [dict(variant="cta"), dict(variant="pipe"),
                                 dict(variant="stream", cluster=4)])
def test_deep_rejects_uncompiled_shapes(cfg):
    """One CTA per token and the pipelined kernel are not compiled for deep
    banks, and their streaming shape takes at most 128 threads (cluster 4
    would need 224 at H = 7168)."""
    inp = wl.make_inputs(4, 13, H, seed=5700)
    d = inp.to("cuda")
    out, newp = torch.empty_like(d.prefix), torch.empty_like(d.prefix)
    with pytest.raises(binding.AttnResError) as e:
        binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out, newp,
                                    config=binding.make_config(**cfg))
    assert e.value.status == -8


def test_deep_bank_limit():
    inp = wl.make_inputs(2, 32, 64, seed=5800)
    d = inp.to("cuda")
    out, newp = torch.empty_like(d.prefix), torch.empty_like(d.prefix)
    with pytest.raises(binding.AttnResError) as e:
        binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out, newp)
    assert e.value.status == -2
