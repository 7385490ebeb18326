"""The 25-layer decoder chain with deferred MoE tails, on the oracle (no GPU).

TensorRT-LLM PR #20546, section "Test Coverage": a 25-layer chain with
deferred MoE tails must be bitwise equal to the eager chain, including the
snapshot bank and a capture tap; section "Model": the prefix sum written to
the bank or carried on is bitwise the same as without the fold.

Fused: layer l calls the op with (P, routed_{l-1}, shared_{l-1}).
Eager: PyTorch adds routed + shared in BF16 first, then the op runs with one
addend.  P <- new_prefix; after every odd layer up to 21 a copy of P joins
the bank (N grows 1 -> 12); every layer's out is the tap."""
import numpy as np
import pytest
import torch

from kimi_k3_attention_gb300 import workloads as wl
from oracle import attnres_add_rmsnorm


def _u(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def run_chain_oracle(H=256, M=4, layers=25, fused=True, last_append=21):
    torch.set_flush_denormal(False)
    emb, p0, L = wl.chain_inputs(M=M, H=H, layers=layers)
    bank = [_u(emb)]
    P = _u(p0)
    taps, prefixes = [], []
    for li, layer in enumerate(L):
        if fused:
            a, a2 = _u(layer.routed), _u(layer.shared)
        else:
            a, a2 = _u(layer.routed + layer.shared), None
        newp, out, _ = attnres_add_rmsnorm(P, a, a2, np.stack(bank), _u(layer.w), _u(layer.gamma), wl.EPS)
        P = newp
        taps.append(out)
        prefixes.append(newp)
        if wl.chain_appends_after(li, last_append):
            bank.append(P.copy())
    return np.stack(bank), prefixes, taps


def test_chain_schedule_grows_bank_to_twelve():
    n = 1
    ns = []
    for li in range(25):
        ns.append(n)
        if wl.chain_appends_after(li):
            n += 1
    assert ns[0] == 1 and ns[-1] == 12 and ns[22:] == [12, 12, 12]


def test_deep_chain_schedule_grows_bank_to_thirty_one():
    n = 1
    for li in range(61):
        if wl.chain_appends_after(li, 59):
            n += 1
    assert n == 31


@pytest.mark.parametrize("layers,last_append,depth", [(25, 21, 12), (61, 59, 31)])
def test_chain_fused_equals_eager_bitwise(layers, last_append, depth):
    bank_f, p_f, t_f = run_chain_oracle(fused=True, layers=layers, last_append=last_append)
    bank_e, p_e, t_e = run_chain_oracle(fused=False, layers=layers, last_append=last_append)
    assert bank_f.shape[0] == depth
    assert (bank_f == bank_e).all()
    for a, b in zip(p_f, p_e):
        assert (a == b).all()
    for a, b in zip(t_f, t_e):
        np.testing.assert_array_equal(a, b)
