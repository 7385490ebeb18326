"""GPU parity on FP16 tensors through the C ABI.

The fused window of TensorRT-LLM PR #20546 (section "Model") is BF16; the
library runs the same op on FP16 tensors (every tensor FP16, both fold
additions rounded to FP16), for every N the BF16 path takes.  The oracle
takes the FP16 codec; new_prefix must be bit-exact, out within 2 FP16 ulp
(with the float32 floor)."""
import os

import numpy as np
import pytest
import torch

from kimi_k3_attention_gb300 import binding
from kimi_k3_attention_gb300 import workloads as wl
from oracle import attnres_add_rmsnorm as oracle_op
from oracle import attnres_rmsnorm as oracle_alone
from oracle import check_out, fold, fp16_decode

from gpu_helpers import Guarded, assert_parity, cfg_name, run_gpu, u16

pytestmark = pytest.mark.gpu

H = wl.H_MODEL
F16 = torch.float16


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def _ceil(a, b):
    return -(-a // b)


def fp16_configs(H):
    """The automatic choice and every cluster size of the split (<= 256
    threads) and streaming (<= 224 threads) shapes that fits this H."""
    need = [_ceil(_ceil(H // 8, c), 32) * 32 for c in range(17)[1:]]
    return ([None] + [binding.make_config("cluster", cluster=c) for c, t in enumerate(need, 1) if t <= 256]
            + [binding.make_config("stream", cluster=c) for c, t in enumerate(need, 1) if t <= 224])


def _t16(bits, shape):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16).copy()).view(F16).view(*shape)


@pytest.mark.parametrize("N", [0, 1, 5, 12])
@pytest.mark.parametrize("M", [1, 8, 32, 64, 300])
@pytest.mark.parametrize("add2", [True, False])
def test_fp16_parity_auto(M, N, add2):
    inp = wl.make_inputs(M, N, H, seed=6000 + 64 * M + N, add2=add2, dtype=F16)
    np_, out = run_gpu(inp)
    assert_parity(inp, np_, out, label=f"M={M} N={N} add2={add2}")


@pytest.mark.parametrize("N", [3, 12])
def test_fp16_every_cluster_size(N):
    inp = wl.make_inputs(5, N, H, seed=6100 + N, dtype=F16)
    ref = None
    for cfg in fp16_configs(H):
        np_, out = run_gpu(inp, config=cfg)
        assert_parity(inp, np_, out, label=f"N={N} {cfg_name(cfg)}")
        if ref is None:
            ref = np_
        assert (np_ == ref).all()


@pytest.mark.parametrize("Hr,N", [(8, 12), (1000, 7), (7176, 12)])
def test_fp16_ragged_width(Hr, N):
    inp = wl.make_inputs(3, N, Hr, seed=6200 + Hr + N, dtype=F16)
    for cfg in fp16_configs(Hr):
        np_, out = run_gpu(inp, config=cfg)
        assert_parity(inp, np_, out, label=f"H={Hr} N={N} {cfg_name(cfg)}")


def test_fp16_golden_fold_cases_on_gpu(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "fold_cases_fp16.txt")):
        if line.strip() and not line.startswith("#"):
            rows.append([int(x, 16) for x in line.split()[:4]])
    rows = np.array(rows, dtype=np.uint16)
    n = len(rows)
    Hs = 8 * ((n + 7) // 8)
    cols = [np.zeros(Hs, np.uint16) for _ in range(4)]
    for c, v in zip(cols, rows.T):
        c[:n] = v
    p, a, a2, e = cols
    inp = wl.make_inputs(1, 1, Hs, seed=3, dtype=F16)
    inp.prefix, inp.add, inp.add2 = _t16(p, (1, Hs)), _t16(a, (1, Hs)), _t16(a2, (1, Hs))
    for cfg in (None, binding.make_config("cluster", cluster=1), binding.make_config("stream", cluster=1)):
        gnp, _ = run_gpu(inp, cfg)
        assert (gnp[0, :n] == e[:n]).all(), [hex(x) for x in gnp[0, :n]]


def test_fp16_fold_sweep_all_patterns():
    """Every finite FP16 add against 64 add2 patterns (all exponents, both
    signs, subnormals), with prefix zero and random: bit-exact to the oracle,
    overflow to infinity included."""
    allb = np.arange(65536, dtype=np.uint16)
    allb = allb[np.isfinite(fp16_decode(allb))]
    rng = np.random.default_rng(19)
    picks = np.concatenate([np.arange(0, 0x7C00, 0x7C00 // 24, dtype=np.uint16)[:24],
                            rng.integers(1, 1024, 8).astype(np.uint16)])
    picks = np.concatenate([picks, picks | 0x8000])
    Hs = 8192
    M = -(-allb.size * picks.size // Hs)
    total = M * Hs
    a = np.resize(allb, total).astype(np.uint16)
    a2 = np.repeat(picks, -(-total // picks.size))[:total].astype(np.uint16)
    for prefix_kind in ("zero", "random"):
        if prefix_kind == "zero":
            p = np.zeros(total, np.uint16)
        else:
            p = rng.integers(0, 65536, total).astype(np.uint16)
            p = np.where(np.isfinite(fp16_decode(p)), p, 0).astype(np.uint16)
        ref, _ = fold(p, a, a2, "fp16")
        inp = wl.make_inputs(M, 1, Hs, seed=5, dtype=F16)
        inp.prefix, inp.add, inp.add2 = _t16(p, (M, Hs)), _t16(a, (M, Hs)), _t16(a2, (M, Hs))
        inp.bank.zero_()
        d = inp.to("cuda")
        out, newp = torch.empty_like(d.prefix), torch.empty_like(d.prefix)
        binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out, newp)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        gnp = u16(newp).ravel()
        bad = np.flatnonzero(gnp != ref)
        assert bad.size == 0, (prefix_kind, hex(p[bad[0]]), hex(a[bad[0]]), hex(a2[bad[0]]),
                               hex(gnp[bad[0]]), hex(ref[bad[0]]))


def test_fp16_subnormal_and_cancelling_addends():
    """A quarter of the positions get FP16 subnormal addends (mantissa 1..1023)
    or near-cancelling pairs; the prefix there is +-0 or subnormal, so the
    subnormal sums reach new_prefix."""
    M, N = 32, 12
    rng = np.random.default_rng(29)
    inp = wl.make_inputs(M, N, H, seed=6300, dtype=F16)
    P = M * H
    p, a, a2 = (u16(x).ravel().copy() for x in (inp.prefix, inp.add, inp.add2))
    pos = rng.permutation(P)[: P // 4]
    sub, can = pos[: len(pos) // 2], pos[len(pos) // 2:]
    rs = lambda n: (rng.integers(1, 1024, n) | (rng.integers(0, 2, n) << 15)).astype(np.uint16)  # noqa: E731
    a[sub], a2[sub], p[sub] = rs(len(sub)), rs(len(sub)), rs(len(sub))
    a2[can] = ((a[can].astype(np.int64) ^ 0x8000) + rng.integers(-2, 3, len(can))).clip(0, 0xFFFF)
    p[can] = (rng.integers(0, 2, len(can)) << 15).astype(np.uint16)
    inp.prefix, inp.add, inp.add2 = _t16(p, (M, H)), _t16(a, (M, H)), _t16(a2, (M, H))
    gnp, gout = run_gpu(inp)
    assert_parity(inp, gnp, gout)
    subn = ((gnp & 0x7C00) == 0) & ((gnp & 0x3FF) != 0)
    assert subn.sum() > 1000


def test_fp16_deterministic_and_add2_equals_presummed():
    inp = wl.make_inputs(16, 9, H, seed=6400, dtype=F16)
    a = run_gpu(inp)
    b = run_gpu(inp)
    assert (a[0] == b[0]).all() and (a[1] == b[1]).all()
    s = (inp.add.float() + inp.add2.float()).to(F16)
    c = run_gpu(wl.Inputs(inp.prefix, s, None, inp.bank, inp.w, inp.gamma, inp.eps))
    assert (a[0] == c[0]).all() and (a[1] == c[1]).all()


@pytest.mark.parametrize("M,N", [(1, 0), (8, 12), (200, 6)])
def test_fp16_alone_and_tap(M, N):
    inp = wl.make_inputs(M, N, H, seed=6500 + M + N, dtype=F16)
    d = inp.to("cuda")
    out, hout = Guarded((M, H), dtype=F16), Guarded((M, H), dtype=F16)
    binding.launch(d.prefix, None, None, d.bank, d.w, d.gamma, d.eps, out.t, None, h_out=hout.t,
                   fold=False)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert out.guards_intact() and hout.guards_intact()
    ref_out, bound, h, hb = oracle_alone(u16(inp.prefix), u16(inp.bank), u16(inp.w), u16(inp.gamma),
                                         inp.eps, with_h=True, fmt="fp16")
    assert check_out(u16(out.t), ref_out, bound, "fp16")["ok"]
    assert check_out(u16(hout.t), h, hb, "fp16")["ok"]

    out2, newp, hout2 = (Guarded((M, H), dtype=F16) for _ in range(3))
    binding.attnres_add_rmsnorm_tap(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps,
                                    out2.t, newp.t, hout2.t)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert out2.guards_intact() and newp.guards_intact() and hout2.guards_intact()
    ref_np, ref_out, bound, h, hb = oracle_op(u16(inp.prefix), u16(inp.add), u16(inp.add2),
                                              u16(inp.bank), u16(inp.w), u16(inp.gamma), inp.eps,
                                              with_h=True, fmt="fp16")
    assert (u16(newp.t) == ref_np).all()
    assert check_out(u16(out2.t), ref_out, bound, "fp16")["ok"]
    assert check_out(u16(hout2.t), h, hb, "fp16")["ok"]


@pytest.mark.parametrize("cfg", [dict(variant="cta"), dict(variant="pipe")])
def test_fp16_rejects_uncompiled_shapes(cfg):
    inp = wl.make_inputs(4, 3, H, seed=6600, dtype=F16)
    d = inp.to("cuda")
    out, newp = torch.empty_like(d.prefix), torch.empty_like(d.prefix)
    with pytest.raises(binding.AttnResError) as e:
        binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out, newp,
                                    config=binding.make_config(**cfg))
    assert e.value.status == -8


@pytest.mark.parametrize("N", [13, 20, 23, 31])
@pytest.mark.parametrize("M", [1, 64, 300])
def test_fp16_deep_banks(M, N):
    """FP16 tensors with more than 12 snapshots: the deep split shape up to 32
    tokens, the deep streaming shape (shared-memory rows from N = 23) above."""
    inp = wl.make_inputs(M, N, H, seed=6700 + M + N, dtype=F16)
    np_, out = run_gpu(inp)
    assert_parity(inp, np_, out, label=f"M={M} N={N}")
    np2, out2 = run_gpu(inp, config=binding.make_config("stream", cluster=8, grid_tokens=7))
    assert_parity(inp, np2, out2, label=f"stream M={M} N={N}")


def test_mixed_dtypes_rejected_by_the_binding():
    inp = wl.make_inputs(2, 1, 64, seed=6800, dtype=F16)
    d = inp.to("cuda")
    out, newp = torch.empty_like(d.prefix), torch.empty_like(d.prefix)
    with pytest.raises(TypeError):
        binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w.to(torch.bfloat16), d.gamma,
                                    d.eps, out, newp)
