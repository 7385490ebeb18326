"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on the
seeded workloads: new_prefix bit-exact, out within the tolerance of
oracle/tolerance.py (2 BF16 ulp with a 2^-16 floor; |delta| <= 1.5e-2 where
|out| <= 4)."""
import math
import os

import numpy as np
import pytest
import torch

from kimi_k3_attention_gb300 import binding
from kimi_k3_attention_gb300 import workloads as wl
from oracle import bf16_decode, fold

from gpu_helpers import Guarded, assert_parity, cfg_name, run_gpu, split_configs, u16

pytestmark = pytest.mark.gpu

H = wl.H_MODEL


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


# ---------------------------------------------------------------- PR reference case

@pytest.mark.parametrize("cfg", split_configs(H), ids=cfg_name)
def test_pr_reference_case_every_variant(cfg):
    inp = wl.pr_reference_case()
    gnp, gout = run_gpu(inp, cfg)
    assert_parity(inp, gnp, gout, label=cfg_name(cfg))


# ---------------------------------------------------------------- decode sweep

@pytest.mark.parametrize("case", list(wl.decode_sweep_cases()), ids=lambda c: f"M{c[1]}-N{c[2]}-{'add2' if c[3] else 'noadd2'}")
def test_decode_sweep_auto(case):
    idx, M, N, has_add2 = case
    inp = wl.decode_sweep_inputs(idx, M, N, has_add2)
    gnp, gout = run_gpu(inp)
    assert_parity(inp, gnp, gout, label=f"case {idx}")


# the automatic cluster size of the register-capped split shape, per M, for
# tokens of at least 9 rows up to M = 28; otherwise about 128 / M (4 from 29)
SPLIT2_CLUSTER = {17: 4, 18: 4, 19: 6, 20: 6, 21: 6, 22: 6, 23: 6, 24: 5, 25: 5, 26: 8, 27: 8,
                  28: 8, 29: 4, 30: 4, 31: 4, 32: 4}


@pytest.mark.parametrize("M", sorted(SPLIT2_CLUSTER))
def test_decode_auto_every_M_17_to_32(M):
    """Every token count of the register-capped split shape with its
    automatic cluster size (4 to 8 CTAs of 224 to 112 threads), with and
    without add2: parity with the oracle."""
    for N, add2 in ((12, True), (9, False), (3, False)):
        rows = N + (3 if add2 else 2)
        want = (SPLIT2_CLUSTER[M] if rows >= 9
                else min(8, max(4, (128 + M // 2) // M)))
        plan = binding.attnres_plan(M, N, H, has_add2=add2)
        assert plan["variant"] == 5 and plan["cluster"] == want, (N, add2, plan)
        inp = wl.make_inputs(M, N, H, seed=300 + M + N, add2=add2)
        gnp, gout = run_gpu(inp)
        assert_parity(inp, gnp, gout, label=f"M={M} N={N}")


@pytest.mark.parametrize("cfg", split_configs(H)[1:], ids=cfg_name)
@pytest.mark.parametrize("M,N", [(1, 12), (32, 12), (16, 5), (8, 1)])
def test_decode_every_variant(cfg, M, N):
    inp = wl.make_inputs(M, N, H, seed=77 + M + N, add2=True)
    gnp, gout = run_gpu(inp, cfg)
    assert_parity(inp, gnp, gout, label=cfg_name(cfg))


# ---------------------------------------------------------------- bit-exactness stress

@pytest.mark.parametrize("special_prefix", [False, True])
@pytest.mark.parametrize("cfg", [None, binding.make_config("cluster", cluster=4),
                                 binding.make_config("stream", cluster=4),
                                 binding.make_config("pipe", cluster=4),
                                 binding.make_config("cta")], ids=cfg_name)
def test_bit_exact_stress(special_prefix, cfg):
    inp = wl.stress_inputs(special_prefix=special_prefix)
    gnp, gout = run_gpu(inp, cfg)
    assert_parity(inp, gnp, gout)
    if special_prefix:
        # subnormal sums must reach the updated prefix (exponent field 0, non-zero)
        sub = ((gnp & 0x7F80) == 0) & ((gnp & 0x7F) != 0)
        assert sub.sum() > 1000


def test_golden_fold_cases_on_gpu(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "fold_cases.txt")):
        if line.strip() and not line.startswith("#"):
            rows.append([int(x, 16) for x in line.split()[:4]])
    rows = np.array(rows, dtype=np.uint16)
    n = len(rows)
    Hs = 8 * ((n + 7) // 8)
    p = np.zeros(Hs, np.uint16)
    a = np.zeros(Hs, np.uint16)
    a2 = np.zeros(Hs, np.uint16)
    e = np.zeros(Hs, np.uint16)
    p[:n], a[:n], a2[:n], e[:n] = rows.T
    t = lambda x: torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16)  # noqa: E731
    inp = wl.make_inputs(1, 1, Hs, seed=3)
    inp.prefix, inp.add, inp.add2 = t(p)[None], t(a)[None], t(a2)[None]
    for cfg in (None, binding.make_config("cta"), binding.make_config("cluster", cluster=1)):
        gnp, _ = run_gpu(inp, cfg)
        assert (gnp[0, :n] == e[:n]).all(), [hex(x) for x in gnp[0, :n]]


def test_fold_sweep_all_patterns():
    """Every finite BF16 add against 64 add2 patterns (all exponents, both
    signs, subnormals), with prefix zero and random: bit-exact to the oracle."""
    allb = np.arange(65536, dtype=np.uint16)
    allb = allb[np.isfinite(bf16_decode(allb))]
    rng = np.random.default_rng(9)
    picks = np.concatenate([np.arange(0, 0x7F80, 0x7F80 // 24, dtype=np.uint16)[:24],
                            rng.integers(1, 128, 8).astype(np.uint16)])
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
            p = np.where(np.isfinite(bf16_decode(p)), p, 0).astype(np.uint16)
        ref, _ = fold(p, a, a2)
        ok = np.isfinite(bf16_decode(ref))
        t = lambda x: torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).view(M, Hs)  # noqa: E731
        inp = wl.make_inputs(M, 1, Hs, seed=5)
        inp.prefix, inp.add, inp.add2 = t(p), t(a), t(a2)
        inp.bank.zero_()
        gnp, _ = run_gpu(inp)
        bad = np.flatnonzero((gnp.ravel() != ref) & ok)
        assert bad.size == 0, (prefix_kind, hex(p[bad[0]]), hex(a[bad[0]]), hex(a2[bad[0]]),
                               hex(gnp.ravel()[bad[0]]), hex(ref[bad[0]]))


# ---------------------------------------------------------------- 25-layer chain

def _chain_gpu(fused, M=8, layers=25, last_append=21):
    emb, p0, layers = wl.chain_inputs(M=M, layers=layers)
    dev = "cuda"
    bank = [emb.to(dev)]
    P = p0.to(dev)
    taps, prefixes = [], []
    for li, L in enumerate(layers):
        w, g = L.w.to(dev), L.gamma.to(dev)
        r, s = L.routed.to(dev), L.shared.to(dev)
        if fused:
            a, a2 = r, s
        else:
            a, a2 = r + s, None          # PyTorch's BF16 addition first
        b = torch.stack(bank).contiguous()
        out = torch.empty_like(P)
        newp = torch.empty_like(P)
        binding.attnres_add_rmsnorm(P, a, a2, b, w, g, wl.EPS, out, newp)
        P = newp
        taps.append(u16(out))
        prefixes.append(u16(newp))
        if wl.chain_appends_after(li, last_append):
            bank.append(P.clone())
    torch.cuda.synchronize()
    return u16(torch.stack(bank)), prefixes, taps


@pytest.mark.parametrize("layers,last_append,depth", [(25, 21, 12), (61, 59, 31)])
def test_chain_fused_equals_eager_bitwise_and_oracle(layers, last_append, depth):
    """The 25-layer chain of the pages (bank 1 -> 12), and a 61-layer chain
    whose bank grows to 31 snapshots (the deep-bank kernels in the hand-off)."""
    bf, pf, tf = _chain_gpu(True, layers=layers, last_append=last_append)
    be, pe, te = _chain_gpu(False, layers=layers, last_append=last_append)
    assert bf.shape[0] == depth
    assert (bf == be).all()
    for a, b in zip(pf, pe):
        assert (a == b).all()
    for a, b in zip(tf, te):
        assert (a == b).all()
    # and layer by layer against the oracle on the same inputs
    from oracle import attnres_add_rmsnorm as oop, check_out
    emb, p0, chain = wl.chain_inputs(M=8, layers=layers)
    bank = [u16(emb)]
    P = u16(p0)
    for li, L in enumerate(chain):
        npb, out, bound = oop(P, u16(L.routed), u16(L.shared), np.stack(bank), u16(L.w),
                              u16(L.gamma), wl.EPS)
        assert (npb == pf[li]).all(), li
        r = check_out(tf[li], out, bound)
        assert r["ok"], (li, r)
        P = npb
        if wl.chain_appends_after(li, last_append):
            bank.append(P.copy())


# ---------------------------------------------------------------- invariants on the GPU

@pytest.mark.parametrize("cfg", [None, binding.make_config("cta"),
                                 binding.make_config("cluster", cluster=16)], ids=cfg_name)
def test_two_addends_equal_one_presummed_addend(cfg):
    """Section "Test Coverage": two addends give bitwise the same updated
    prefix sum and output as one addend holding their BF16 sum."""
    for M, N in ((1, 1), (8, 7), (16, 12), (32, 3)):
        inp = wl.make_inputs(M, N, H, seed=500 + M * 13 + N, add2=True)
        gnp2, gout2 = run_gpu(inp, cfg)
        pre = wl.Inputs(inp.prefix, inp.add + inp.add2, None, inp.bank, inp.w, inp.gamma, inp.eps)
        gnp1, gout1 = run_gpu(pre, cfg)
        assert (gnp1 == gnp2).all() and (gout1 == gout2).all()
        # and the same prefix as PyTorch's prefix + (routed + shared)
        assert (u16(inp.prefix + (inp.add + inp.add2)) == gnp2).all()


def test_deterministic_repeats():
    inp = wl.make_inputs(32, 12, H, seed=42).to("cuda")
    outs = []
    for _ in range(5):
        out = torch.empty_like(inp.prefix)
        newp = torch.empty_like(inp.prefix)
        binding.attnres_add_rmsnorm(inp.prefix, inp.add, inp.add2, inp.bank, inp.w, inp.gamma,
                                    inp.eps, out, newp)
        outs.append((u16(out), u16(newp)))
    for o in outs[1:]:
        assert (o[0] == outs[0][0]).all() and (o[1] == outs[0][1]).all()


def test_all_split_cluster_sizes_agree_on_new_prefix():
    inp = wl.make_inputs(16, 9, H, seed=43)
    ref = None
    for cfg in split_configs(H):
        gnp, _ = run_gpu(inp, cfg)
        if ref is None:
            ref = gnp
        assert (gnp == ref).all(), cfg_name(cfg)


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("Hs", [8, 16, 24, 64, 72, 1000, 2056, 7176, 8192, 16384])
def test_ragged_and_small_hidden_sizes(Hs):
    for M, N, add2 in ((1, 1, True), (3, 12, False), (5, 4, True)):
        inp = wl.make_inputs(M, N, Hs, seed=Hs + M + N, add2=add2)
        for cfg in split_configs(Hs):
            gnp, gout = run_gpu(inp, cfg)
            assert_parity(inp, gnp, gout, label=f"H={Hs} {cfg_name(cfg)}")


@pytest.mark.parametrize("grid_tokens", [1, 3, 64])
def test_token_loop(grid_tokens):
    """Fewer token CTAs than tokens: each cluster loops over tokens."""
    inp = wl.make_inputs(67, 6, H, seed=11)
    for variant, cl in (("cluster", 4), ("cluster", 8), ("stream", 4), ("pipe", 4), ("pipe", 7)):
        cfg = binding.make_config(variant, cluster=cl, grid_tokens=grid_tokens)
        gnp, gout = run_gpu(inp, cfg)
        assert_parity(inp, gnp, gout)
    gnp, gout = run_gpu(inp, binding.make_config("cta", grid_tokens=grid_tokens))
    assert_parity(inp, gnp, gout)


@pytest.mark.parametrize("grid_tokens,tail_tokens", [(2, 1), (10, 4), (67, 66), (40, 39), (67, 1)])
def test_tail_tokens(grid_tokens, tail_tokens):
    """The last tail_tokens clusters take one token each, the others walk the
    rest: every token once, the same bits as one cluster per token."""
    inp = wl.make_inputs(67, 6, H, seed=13)
    for variant, cl in (("stream", 7), ("stream", 4), ("stream", 8), ("stream", 5)):
        plain = binding.make_config(variant, cluster=cl, grid_tokens=67)
        walk = binding.make_config(variant, cluster=cl, grid_tokens=grid_tokens,
                                   tail_tokens=tail_tokens)
        rnp, rout = run_gpu(inp, plain)
        gnp, gout = run_gpu(inp, walk)
        assert (gnp == rnp).all() and (gout == rout).all(), (variant, cl)
        assert_parity(inp, gnp, gout, label=f"{variant}{cl}")


@pytest.mark.parametrize("M,N", [(300, 3), (1200, 12), (2500, 1)])
def test_automatic_walk(M, N):
    """Register-capped shape with the launch-time grid (walking clusters and
    one-token clusters at the end): the same bits as one cluster per token."""
    inp = wl.make_inputs(M, N, H, seed=14 + M, add2=True)
    plan = binding.attnres_plan(M, N, H)
    assert plan["variant"] == 3 and plan["grid_tokens"] == 0 and plan["tail_tokens"] == 0
    gnp, gout = run_gpu(inp)
    rnp, rout = run_gpu(inp, binding.make_config("stream", cluster=plan["cluster"], grid_tokens=M))
    assert (gnp == rnp).all() and (gout == rout).all()
    toks = np.unique(np.linspace(0, M - 1, 64).astype(int))
    assert_parity(inp, gnp, gout, tokens=toks)


@pytest.mark.parametrize("M,N,fp16", [(1500, 16, False), (900, 24, False), (700, 31, False),
                                       (1200, 12, True), (600, 20, True)])
def test_automatic_walk_deep_and_fp16(M, N, fp16):
    """The launch-time walk of the deep streaming shapes and of FP16 tensors:
    the same bits as one cluster per token, parity with the oracle."""
    inp = wl.make_inputs(M, N, H, seed=16 + M + N, add2=True,
                         dtype=torch.float16 if fp16 else torch.bfloat16)
    plan = binding.attnres_plan(M, N, H)
    assert plan["variant"] == 3 and plan["grid_tokens"] == 0
    gnp, gout = run_gpu(inp)
    rnp, rout = run_gpu(inp, binding.make_config("stream", cluster=plan["cluster"], grid_tokens=M))
    assert (gnp == rnp).all() and (gout == rout).all()
    toks = np.unique(np.linspace(0, M - 1, 40).astype(int))
    assert_parity(inp, gnp, gout, tokens=toks)


def test_tail_tokens_rejected():
    inp = wl.make_inputs(9, 2, H, seed=15).to("cuda")
    out, np_ = torch.empty_like(inp.prefix), torch.empty_like(inp.prefix)
    def call(cfg):
        with pytest.raises(binding.AttnResError):
            binding.attnres_add_rmsnorm(inp.prefix, inp.add, inp.add2, inp.bank, inp.w, inp.gamma,
                                        inp.eps, out, np_, config=cfg)
    call(binding.make_config("stream", cluster=4, grid_tokens=4, tail_tokens=4))    # no walker
    call(binding.make_config("stream", cluster=4, grid_tokens=10, tail_tokens=2))   # grid > M
    call(binding.make_config("stream", cluster=4, tail_tokens=2))                   # auto grid
    call(binding.make_config("stream", cluster=4, grid_tokens=4, tail_tokens=-1))
    call(binding.make_config("pipe", cluster=4, grid_tokens=4, tail_tokens=1))
    for v in ("cluster", "cluster2", "cta"):                                       # latency shapes
        call(binding.make_config(v, grid_tokens=4, tail_tokens=1))


def test_more_tokens_than_grid_limit():
    """M above 65535: the grid's token axis is capped and clusters loop."""
    M, Hs = 70000, 64
    inp = wl.make_inputs(M, 2, Hs, seed=12, device="cuda")
    gnp, gout = run_gpu(inp)
    toks = np.array([0, 1, 65534, 65535, 65536, 69999])
    assert_parity(inp, gnp, gout, tokens=toks)


def test_in_place_prefix_and_bank_slot_target():
    inp = wl.make_inputs(8, 5, H, seed=21)
    ref_np, ref_out = run_gpu(inp)
    d = inp.to("cuda")
    # in place: new_prefix is prefix
    P = d.prefix.clone()
    out = torch.empty_like(P)
    binding.attnres_add_rmsnorm(P, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out, P)
    torch.cuda.synchronize()
    assert (u16(P) == ref_np).all() and (u16(out) == ref_out).all()
    # new_prefix written straight into bank slot N of a bank with N+1 slots
    big = torch.empty((6, 8, H), dtype=torch.bfloat16, device="cuda")
    big[:5] = d.bank
    out2 = torch.empty_like(P)
    binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, big[:5], d.w, d.gamma, d.eps, out2, big[5])
    torch.cuda.synchronize()
    assert (u16(big[5]) == ref_np).all() and (u16(out2) == ref_out).all()


def test_side_stream_and_plan():
    inp = wl.make_inputs(16, 12, H, seed=31)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gnp, gout = run_gpu(inp, stream=s)
    assert_parity(inp, gnp, gout)
    for M in (1, 8, 16, 32, 8192):
        plan = binding.attnres_plan(M, 12, H)
        assert plan["variant"] in (1, 2, 3, 4, 5) and plan["threads"] % 32 == 0


def test_invalid_config_rejected_on_device():
    d = wl.make_inputs(4, 3, H, seed=1).to("cuda")
    out = torch.empty_like(d.prefix)
    newp = torch.empty_like(d.prefix)
    for cfg in (binding.make_config("cluster", cluster=17), binding.make_config("cluster", cluster=1),
                binding.make_config("cta", cluster=2), binding.make_config(7),
                binding.make_config("cluster", cluster=8, threads=100)):
        with pytest.raises(binding.AttnResError) as e:
            binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps,
                                        out, newp, config=cfg)
        assert e.value.status == -8


def test_subnormal_inputs_in_the_mixture():
    """All sources tiny (BF16 subnormal scale): outputs stay finite and within
    tolerance (the norms divide by sqrt(mean + eps))."""
    inp = wl.make_inputs(4, 3, H, seed=8)
    for name in ("prefix", "add", "add2"):
        setattr(inp, name, (getattr(inp, name).float() * 1e-39).to(torch.bfloat16))
    inp.bank = (inp.bank.float() * 1e-39).to(torch.bfloat16)
    gnp, gout = run_gpu(inp)
    assert_parity(inp, gnp, gout)


# ---------------------------------------------------------------- full size, sampled

def test_bandwidth_config_sampled():
    """M=8192, N=12, H=7168, add2 present, in the automatic launch
    configuration the benchmark times: new_prefix checked for every token
    against the oracle's fold, out for 48 sampled tokens."""
    inp = wl.bandwidth_inputs(device="cuda")
    gnp, gout = run_gpu(inp)
    P, A, A2 = u16(inp.prefix), u16(inp.add), u16(inp.add2)
    for t0 in range(0, inp.M, 1024):
        ref, _ = fold(P[t0:t0 + 1024], A[t0:t0 + 1024], A2[t0:t0 + 1024])
        assert (gnp[t0:t0 + 1024] == ref).all(), t0
    rng = np.random.default_rng(0)
    toks = np.unique(np.concatenate([[0, 1, 151, 152, 4095, 8190, 8191], rng.integers(0, 8192, 41)]))
    cpu = inp.to("cpu")
    assert_parity(cpu, gnp, gout, tokens=toks)


@pytest.mark.parametrize("M", [1, 32, 300])
def test_pdl_on_and_off_identical(M):
    """Programmatic dependent launch changes scheduling only."""
    inp = wl.make_inputs(M, 12, H, seed=61 + M)
    on = run_gpu(inp, binding.make_config(pdl=1))
    off = run_gpu(inp, binding.make_config(pdl=-1))
    assert (on[0] == off[0]).all() and (on[1] == off[1]).all()
    assert_parity(inp, *on)


def test_back_to_back_dependent_calls_with_pdl():
    """A chain where each call reads the previous call's new_prefix, queued
    without host synchronisation: the dependency must hold under PDL."""
    inp = wl.make_inputs(8, 4, H, seed=62)
    d = inp.to("cuda")
    P = d.prefix.clone()
    outs = []
    for _ in range(6):
        out = torch.empty_like(P)
        newp = torch.empty_like(P)
        binding.attnres_add_rmsnorm(P, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out, newp,
                                    config=binding.make_config(pdl=1))
        outs.append((newp, out))
        P = newp
    torch.cuda.synchronize()
    from oracle import attnres_add_rmsnorm as oop
    Pc = u16(inp.prefix)
    for newp, out in outs:
        ref_np, _, _ = oop(Pc, u16(inp.add), u16(inp.add2), u16(inp.bank), u16(inp.w),
                           u16(inp.gamma), inp.eps)
        assert (u16(newp) == ref_np).all()
        Pc = ref_np


@pytest.mark.parametrize("stages", [2, 3, 4])
@pytest.mark.parametrize("cl", [4, 8])
@pytest.mark.parametrize("add2", [True, False])
def test_pipe_stages(stages, cl, add2):
    """The pipelined kernel at every ring depth, with the ring wrapping many
    times (few resident clusters, many tokens) and a ragged token count."""
    inp = wl.make_inputs(203, 12, H, seed=70 + stages + cl, add2=add2)
    cfg = binding.make_config("pipe", cluster=cl, stages=stages, grid_tokens=5)
    gnp, gout = run_gpu(inp, cfg)
    assert_parity(inp, gnp, gout, label=f"pipe{cl}s{stages}")
    auto = binding.make_config("pipe", cluster=cl, stages=stages)
    gnp2, gout2 = run_gpu(inp, auto)
    assert (gnp2 == gnp).all() and (gout2 == gout).all()


def test_pipe_invalid_stages_rejected():
    d = wl.make_inputs(4, 12, H, seed=1).to("cuda")
    out = torch.empty_like(d.prefix)
    newp = torch.empty_like(d.prefix)
    for cfg in (binding.make_config("pipe", stages=5), binding.make_config("pipe", stages=1),
                binding.make_config("cluster", cluster=8, stages=2)):
        with pytest.raises(binding.AttnResError) as e:
            binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps,
                                        out, newp, config=cfg)
        assert e.value.status == -8


@pytest.mark.parametrize("prefetch", [-1, 1, 2, 3, 4, 5, 7, 8, 9, 15])
def test_prefetch_modes_identical(prefetch):
    """L2 prefetch and early dependent launch change scheduling only; a
    dependent chain queued without host synchronisation stays exact."""
    inp = wl.make_inputs(16, 6, H, seed=90)
    ref = run_gpu(inp, binding.make_config("cluster", cluster=8, prefetch=-1))
    got = run_gpu(inp, binding.make_config("cluster", cluster=8, prefetch=prefetch))
    assert (ref[0] == got[0]).all() and (ref[1] == got[1]).all()
    d = inp.to("cuda")
    P = d.prefix.clone()
    outs = []
    for _ in range(5):
        out, newp = torch.empty_like(P), torch.empty_like(P)
        binding.attnres_add_rmsnorm(P, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out, newp,
                                    config=binding.make_config("cluster", cluster=8, prefetch=prefetch))
        outs.append(newp)
        P = newp
    torch.cuda.synchronize()
    from oracle import fold
    Pc = u16(inp.prefix)
    for newp in outs:
        Pc, _ = fold(Pc, u16(inp.add), u16(inp.add2))
        assert (u16(newp) == Pc).all()


def _random_cases(n=40, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        H8 = int(rng.choice([1, 3, 8, 40, 100, 257, 896, 897, 1500, 2048]))
        Hs = 8 * H8
        M = int(rng.choice([1, 2, 7, 33, 65, 130]))
        N = int(rng.integers(0, 13))
        add2 = bool(rng.integers(0, 2))
        variant = str(rng.choice(["auto", "cta", "cluster", "stream", "pipe"]))
        lim = {"cta": None, "cluster": 256, "stream": 224, "pipe": 256, "auto": None}[variant]
        cluster = 0
        if lim is not None:
            ok = [c for c in range(1, 17) if -(-(-(-H8 // c)) // 32) * 32 <= lim]
            if not ok:
                continue
            cluster = int(rng.choice(ok))
        if variant == "cta" and -(-(-(-H8 // 2)) // 32) * 32 > 448:
            continue
        gt = int(rng.choice([0, 0, 1, 3]))
        cases.append((M, N, Hs, add2, variant, cluster, gt, int(rng.integers(0, 10 ** 6))))
    return cases


@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: "M{}-N{}-H{}-{}-{}{}-g{}".format(
    c[0], c[1], c[2], "a2" if c[3] else "a1", c[4], c[5], c[6]))
def test_random_configurations(case):
    """Seeded random shapes x variants x cluster sizes x grid strides, N = 0
    included: new_prefix bit-exact, out within tolerance, guards intact."""
    M, N, Hs, add2, variant, cluster, gt, seed = case
    inp = wl.make_inputs(M, max(N, 1), Hs, seed=seed, add2=add2)
    if N == 0:
        inp.bank = inp.bank[:0]
    cfg = None if variant == "auto" else binding.make_config(variant, cluster=cluster, grid_tokens=gt)
    gnp, gout = run_gpu(inp, cfg)
    assert_parity(inp, gnp, gout, label=str(case))


def _random_wide_cases(n=40, seed=2612):
    """Deep banks (N up to 31) and FP16 tensors (N up to 31) in the split and
    streaming shapes, with random cluster sizes, grid strides and prefetch
    modes."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        H8 = int(rng.choice([1, 3, 40, 257, 896, 897, 2048]))
        M = int(rng.choice([1, 5, 33, 130]))
        fp16 = bool(rng.integers(0, 2))
        N = int(rng.integers(0, 32)) if fp16 else int(rng.integers(13, 32))
        add2 = bool(rng.integers(0, 2))
        variant = str(rng.choice(["auto", "cluster", "stream"]))
        lim = {"cluster": 256, "stream": 224 if N <= 12 else 128, "auto": None}[variant]
        cluster = 0
        if lim is not None:
            ok = [c for c in range(1, 17) if -(-(-(-H8 // c)) // 32) * 32 <= lim]
            if not ok:
                continue
            cluster = int(rng.choice(ok))
        gt = int(rng.choice([0, 0, 1, 3]))
        pf = int(rng.choice([0, -1, 1, 4, 5])) if variant != "auto" else 0
        cases.append((M, N, 8 * H8, add2, fp16, variant, cluster, gt, pf, int(rng.integers(0, 10 ** 6))))
    return cases


@pytest.mark.parametrize("case", _random_wide_cases(), ids=lambda c: "M{}-N{}-H{}-{}-{}-{}{}-g{}-p{}".format(
    c[0], c[1], c[2], "a2" if c[3] else "a1", "f16" if c[4] else "bf16", c[5], c[6], c[7], c[8]))
def test_random_deep_and_fp16_configurations(case):
    M, N, Hs, add2, fp16, variant, cluster, gt, pf, seed = case
    inp = wl.make_inputs(M, max(N, 1), Hs, seed=seed, add2=add2,
                         dtype=torch.float16 if fp16 else torch.bfloat16)
    if N == 0:
        inp.bank = inp.bank[:0]
    cfg = None if variant == "auto" else binding.make_config(variant, cluster=cluster, grid_tokens=gt,
                                                             prefetch=pf)
    gnp, gout = run_gpu(inp, cfg)
    assert_parity(inp, gnp, gout, label=str(case))


def test_all_zero_sources():
    """Every source zero: sums of squares are 0, the norms divide by sqrt(eps),
    alpha is uniform and out is exactly zero."""
    inp = wl.make_inputs(4, 5, H, seed=91)
    for name in ("prefix", "add", "add2"):
        setattr(inp, name, torch.zeros_like(getattr(inp, name)))
    inp.bank = torch.zeros_like(inp.bank)
    gnp, gout = run_gpu(inp)
    assert_parity(inp, gnp, gout)
    assert ((gout & 0x7FFF) == 0).all()


@pytest.mark.parametrize("scale", [1e15, 1e-30])
def test_large_and_tiny_magnitudes(scale):
    """Magnitudes far from 1 while sum(v^2) stays inside float32's range: the
    RMS normalisations make out scale-free, so it must match the oracle."""
    inp = wl.make_inputs(8, 6, H, seed=92)
    for name in ("prefix", "add", "add2"):
        setattr(inp, name, (getattr(inp, name).float() * scale).to(torch.bfloat16))
    inp.bank = (inp.bank.float() * scale).to(torch.bfloat16)
    gnp, gout = run_gpu(inp)
    assert_parity(inp, gnp, gout)


def test_fold_overflow_to_infinity_is_bit_exact():
    """Sums beyond the largest BF16 round to +-inf in both the fold and the
    oracle; new_prefix stays bit-exact (outputs of such tokens are not finite
    and are not compared)."""
    inp = wl.make_inputs(2, 1, 64, seed=93)
    big = torch.full((2, 64), 3.0e38).to(torch.bfloat16)
    inp.prefix, inp.add, inp.add2 = big.clone(), big.clone(), -big.clone() * 0.5
    inp.add2[:, ::2] = big[:, ::2]
    gnp, _ = run_gpu(inp)
    from oracle import fold
    ref, _ = fold(u16(inp.prefix), u16(inp.add), u16(inp.add2))
    assert (gnp == ref).all()
    assert ((ref & 0x7FFF) == 0x7F80).any()


def test_two_host_threads_two_streams():
    """Calls from two host threads on two streams at once (the library's
    per-device caches are atomics; no device state is shared by calls)."""
    import threading
    cases = [wl.make_inputs(32, 12, H, seed=700), wl.make_inputs(300, 5, H, seed=701)]
    refs = [run_gpu(c) for c in cases]
    results = [None, None]
    errors = []

    def worker(i):
        try:
            d = cases[i].to("cuda")
            s = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(s):
                for _ in range(20):
                    out, newp = torch.empty_like(d.prefix), torch.empty_like(d.prefix)
                    binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma,
                                                d.eps, out, newp, stream=s)
                    outs.append((out, newp))
            s.synchronize()
            results[i] = outs
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    th = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    for i in range(2):
        for out, newp in results[i]:
            assert (u16(newp) == refs[i][0]).all() and (u16(out) == refs[i][1]).all()


def test_cuda_graph_capture_and_replay():
    """The op captured in a CUDA graph (with programmatic dependent launch
    between the captured calls) replays to the same bits."""
    inp = wl.make_inputs(16, 12, H, seed=702)
    ref_np, ref_out = run_gpu(inp)
    d = inp.to("cuda")
    s = torch.cuda.Stream()
    out, newp = torch.empty_like(d.prefix), torch.empty_like(d.prefix)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out, newp,
                                    stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(10):
            binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps, out,
                                        newp, stream=s)
    out.zero_()
    newp.zero_()
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    assert (u16(newp) == ref_np).all() and (u16(out) == ref_out).all()


@pytest.mark.parametrize("prefetch", [-1, 4, 5, 7])
def test_next_token_prefetch_identical(prefetch):
    """Clusters walking several tokens with the next token's rows prefetched
    into L2 (bit 4): same bits as without, parity with the oracle."""
    inp = wl.make_inputs(67, 12, H, seed=95)
    cfg = binding.make_config("stream", cluster=7, grid_tokens=5, prefetch=prefetch)
    got = run_gpu(inp, cfg)
    ref = run_gpu(inp, binding.make_config("stream", cluster=7, grid_tokens=5, prefetch=-1))
    assert (got[0] == ref[0]).all() and (got[1] == ref[1]).all()
    assert_parity(inp, *got)


@pytest.mark.parametrize("eps", [1e-12, 1e-2, 1.0, 1e3])
@pytest.mark.parametrize("cfg", [None, binding.make_config("stream", cluster=7),
                                 binding.make_config("cta")], ids=cfg_name)
def test_eps_range(eps, cfg):
    """eps from negligible to dominant (1e3 >> mean(v^2) = 1: both norms are
    then close to a plain 1/sqrt(eps) scaling); the oracle takes the same
    float32 eps."""
    inp = wl.make_inputs(6, 7, H, seed=900 + round(math.log10(eps)), eps=eps)
    np_, out = run_gpu(inp, config=cfg)
    assert_parity(inp, np_, out, label=f"eps={eps} {cfg_name(cfg)}")
