"""GPU parity of the calls beyond the fused epilogue itself, through the C
ABI: the pre-norm mixture tap, the attention-residual + RMSNorm alone, and
the standalone fold kernel."""
import numpy as np
import pytest
import torch

from kimi_k3_attention_gb300 import binding
from kimi_k3_attention_gb300 import workloads as wl
from oracle import attnres_add_rmsnorm as oracle_op
from oracle import attnres_rmsnorm as oracle_alone
from oracle import check_out, fold

from gpu_helpers import Guarded, assert_parity, run_gpu, u16

pytestmark = pytest.mark.gpu

H = wl.H_MODEL


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def _cfgs():
    return [None, binding.make_config("cluster", cluster=4), binding.make_config("cluster", cluster=8),
            binding.make_config("stream", cluster=7), binding.make_config("stream", cluster=4)]


@pytest.mark.parametrize("M,N", [(1, 1), (8, 12), (32, 5), (300, 12)])
@pytest.mark.parametrize("ci", range(5))
def test_alone_parity(M, N, ci):
    cfg = _cfgs()[ci]
    inp = wl.make_inputs(M, N, H, seed=300 + M + N)
    d = inp.to("cuda")
    out = Guarded((M, H))
    hout = Guarded((M, H))
    binding.launch(d.prefix, None, None, d.bank, d.w, d.gamma, d.eps, out.t, None, h_out=hout.t,
                   fold=False, config=cfg)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert out.guards_intact() and hout.guards_intact()
    ref_out, bound, h, hb = oracle_alone(u16(inp.prefix), u16(inp.bank), u16(inp.w),
                                         u16(inp.gamma), inp.eps, with_h=True)
    r = check_out(u16(out.t), ref_out, bound)
    assert r["ok"], r
    r = check_out(u16(hout.t), h, hb)
    assert r["ok"], r


def test_alone_entry_point_and_rejected_variants():
    inp = wl.make_inputs(16, 7, H, seed=5)
    d = inp.to("cuda")
    out = torch.empty_like(d.prefix)
    binding.attnres_rmsnorm(d.prefix, d.bank, d.w, d.gamma, d.eps, out)
    torch.cuda.synchronize()
    ref_out, bound = oracle_alone(u16(inp.prefix), u16(inp.bank), u16(inp.w), u16(inp.gamma), inp.eps)
    assert check_out(u16(out), ref_out, bound)["ok"]
    for cfg in (binding.make_config("cta"), binding.make_config("pipe")):
        with pytest.raises(binding.AttnResError) as e:
            binding.launch(d.prefix, None, None, d.bank, d.w, d.gamma, d.eps, out, None, fold=False,
                           config=cfg)
        assert e.value.status == -8


@pytest.mark.parametrize("M,N,add2", [(1, 3, True), (8, 12, False), (32, 12, True), (200, 6, True)])
def test_tap_parity(M, N, add2):
    inp = wl.make_inputs(M, N, H, seed=400 + M + N, add2=add2)
    d = inp.to("cuda")
    out, newp, hout = Guarded((M, H)), Guarded((M, H)), Guarded((M, H))
    binding.attnres_add_rmsnorm_tap(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps,
                                    out.t, newp.t, hout.t)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert out.guards_intact() and newp.guards_intact() and hout.guards_intact()
    ref_np, ref_out, bound, h, hb = oracle_op(u16(inp.prefix), u16(inp.add),
                                              None if inp.add2 is None else u16(inp.add2),
                                              u16(inp.bank), u16(inp.w), u16(inp.gamma), inp.eps,
                                              with_h=True)
    assert (u16(newp.t) == ref_np).all()
    assert check_out(u16(out.t), ref_out, bound)["ok"]
    r = check_out(u16(hout.t), h, hb)
    assert r["ok"], r
    # the tap changes nothing else
    gnp, gout = run_gpu(inp)
    assert (gnp == u16(newp.t)).all() and (gout == u16(out.t)).all()


@pytest.mark.parametrize("M,Hs", [(1, 8), (3, 24), (32, 7168), (8192, 7168), (77, 16384)])
@pytest.mark.parametrize("add2", [True, False])
def test_tail_add_bit_exact(M, Hs, add2):
    if M <= 32 and Hs >= 64:   # subnormal and near-cancelling addends, +-0/subnormal prefix
        inp = wl.stress_inputs(M=M, N=1, H=Hs, seed=M + Hs, special_prefix=True)
    else:
        inp = wl.make_inputs(M, 1, Hs, seed=M + Hs, add2=True)
    d = inp.to("cuda")
    newp = Guarded((M, Hs))
    binding.attnres_tail_add(d.prefix, d.add, d.add2 if add2 else None, newp.t)
    torch.cuda.synchronize()
    assert newp.guards_intact()
    ref, _ = fold(u16(inp.prefix), u16(inp.add), u16(inp.add2) if add2 else None)
    assert (u16(newp.t) == ref).all()


def test_tail_add_in_place_matches_fused_prefix():
    inp = wl.stress_inputs(special_prefix=True)
    d = inp.to("cuda")
    P = d.prefix.clone()
    binding.attnres_tail_add(P, d.add, d.add2, P)
    torch.cuda.synchronize()
    gnp, _ = run_gpu(inp)
    assert (u16(P) == gnp).all()


@pytest.mark.parametrize("add2", [True, False])
def test_no_snapshots(add2):
    """N = 0 (the first layer): every variant, bank pointer NULL."""
    from gpu_helpers import split_configs, cfg_name
    from oracle import attnres_add_rmsnorm as oop
    for M in (1, 5, 100):
        inp = wl.make_inputs(M, 1, H, seed=600 + M, add2=add2)
        d = inp.to("cuda")
        ref_np, ref_out, bound = oop(u16(inp.prefix), u16(inp.add),
                                     u16(inp.add2) if add2 else None,
                                     np.zeros((0, M, H), np.uint16), u16(inp.w), u16(inp.gamma),
                                     inp.eps)
        for cfg in split_configs(H):
            out, newp = Guarded((M, H)), Guarded((M, H))
            empty = torch.empty((0, M, H), dtype=torch.bfloat16, device="cuda")
            binding.launch(d.prefix, d.add, d.add2 if add2 else None, empty, d.w, d.gamma, d.eps,
                           out.t, newp.t, M=M, N=0, H=H, config=cfg)
            torch.cuda.synchronize()
            assert binding.device_status() == 0
            assert out.guards_intact() and newp.guards_intact()
            assert (u16(newp.t) == ref_np).all(), cfg_name(cfg)
            assert check_out(u16(out.t), ref_out, bound)["ok"], cfg_name(cfg)
    # no fold, no snapshots: a plain RMSNorm of the prefix
    out = torch.empty_like(d.prefix)
    binding.launch(d.prefix, None, None, None, d.w, d.gamma, d.eps, out, None, M=M, N=0, H=H,
                   fold=False)
    torch.cuda.synchronize()
    ref = torch.nn.functional.rms_norm(inp.prefix.double(), (H,), inp.gamma.double(),
                                       float(np.float32(inp.eps))).numpy()
    assert check_out(u16(out), ref, np.abs(ref) + 1e-30)["ok"]


@pytest.mark.parametrize("M,N,Hs", [(8192, 12, 7168), (5, 3, 7168), (300, 0, 2056), (33, 12, 64)])
def test_access_pattern_measurement_aid(M, N, Hs):
    """attnres_access_pattern (the fused op's traffic without its arithmetic):
    new_prefix is a copy of prefix and out the XOR of the N+3 input rows."""
    g = torch.Generator(device="cuda")
    g.manual_seed(M + N)
    rnd = lambda *sh: torch.randn(sh, generator=g, device="cuda").to(torch.bfloat16)  # noqa: E731
    P, A, A2, B = rnd(M, Hs), rnd(M, Hs), rnd(M, Hs), rnd(N, M, Hs)
    out, newp = Guarded((M, Hs)), Guarded((M, Hs))
    binding.attnres_access_pattern(P, A, A2, B, out.t, newp.t)
    torch.cuda.synchronize()
    assert out.guards_intact() and newp.guards_intact()
    assert (u16(newp.t) == u16(P)).all()
    x = u16(P) ^ u16(A) ^ u16(A2)
    for i in range(N):
        x = x ^ u16(B[i])
    assert (u16(out.t) == x).all()
