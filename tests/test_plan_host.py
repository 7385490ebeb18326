"""The automatic launch configuration without a GPU (attnres_plan_host): the
rule the library documents for each regime of M, restated here and compared
field by field."""
import os

import pytest

from kimi_k3_attention_gb300 import binding
from kimi_k3_attention_gb300.build import LIB

pytestmark = pytest.mark.skipif(not os.path.exists(LIB), reason="libattnres.so not built")

H = 7168
H8 = H // 8
# cluster size per token of the register-capped split shape for 17..28 tokens of
# at least 9 rows (bank, prefix, addends)
SPLIT2 = {17: 4, 18: 4, 19: 6, 20: 6, 21: 6, 22: 6, 23: 6, 24: 5, 25: 5, 26: 8, 27: 8, 28: 8}


def about_128_per_m(M):
    """About 128 CTAs per call: 128 / M rounded, clamped to 4..8."""
    return min(8, max(4, (128 + M // 2) // M))


def threads_for(cluster, chunks_per_thread=1):
    cpc = -(-H8 // cluster)
    return -(-(-(-cpc // chunks_per_thread)) // 32) * 32


@pytest.mark.parametrize("M", range(1, 33))
@pytest.mark.parametrize("N,add2", [(12, True), (9, False), (6, True), (5, True), (3, False), (0, True)])
def test_decode_window(M, N, add2):
    p = binding.attnres_plan_host(M, N, H, has_add2=add2)
    rows = N + (3 if add2 else 2)
    if M <= 16:
        want_variant, want_cluster = 2, about_128_per_m(M)
    else:
        want_variant = 5
        want_cluster = SPLIT2[M] if (M <= 28 and rows >= 9) else about_128_per_m(M)
    assert (p["variant"], p["cluster"]) == (want_variant, want_cluster), (M, N, add2, p)
    assert p["threads"] == threads_for(p["cluster"])
    assert p["grid_tokens"] == M and p["prefetch"] == 9 and p["pdl"] == 1
    assert p["tail_tokens"] == 0 and p["stages"] == 0


@pytest.mark.parametrize("M", [33, 40, 48, 49, 64, 96, 97, 512, 8192, 65536])
def test_beyond_the_decode_window(M):
    p = binding.attnres_plan_host(M, 12, H)
    if M <= 48:
        assert (p["variant"], p["cluster"], p["threads"], p["grid_tokens"]) == (2, 8, 128, M)
        assert p["prefetch"] == 1
    elif M <= 96:
        assert (p["variant"], p["cluster"], p["threads"], p["grid_tokens"]) == (3, 4, 224, 0)
        assert p["prefetch"] == 1 | 4
    else:
        assert (p["variant"], p["cluster"], p["threads"], p["grid_tokens"]) == (3, 7, 128, 0)
        assert p["prefetch"] == 4


@pytest.mark.parametrize("N", [13, 16, 23, 24, 31])
@pytest.mark.parametrize("M", [1, 4, 8, 17, 32, 33, 8192])
def test_deep_banks(M, N):
    """More than 12 snapshots: the uncapped split shape up to 32 tokens (4 CTAs
    from 8 tokens on once N >= 24), their streaming shape of 7 x 128 beyond."""
    p = binding.attnres_plan_host(M, N, H)
    if M <= 32:
        want = 4 if (N >= 24 and M >= 8) else about_128_per_m(M)
        assert (p["variant"], p["cluster"]) == (2, want)
        assert p["grid_tokens"] == M
    else:
        assert (p["variant"], p["cluster"], p["threads"], p["grid_tokens"]) == (3, 7, 128, 0)


def test_other_hidden_sizes_scale_the_cluster():
    """The cluster sizes are for H = 7168 and scale with H (at least as many CTAs
    as 256 threads of 8 columns need)."""
    p = binding.attnres_plan_host(1, 12, 16384)
    assert p["variant"] == 2 and p["cluster"] == 16 and p["threads"] == 128
    p = binding.attnres_plan_host(1, 12, 1024)
    assert p["variant"] == 2 and p["cluster"] == 1 and p["threads"] == 128


def test_rejects_bad_shapes():
    for M, N, Hs in ((0, 3, H), (1, 32, H), (1, 3, 12), (1, 3, 16392)):
        with pytest.raises(binding.AttnResError):
            binding.attnres_plan_host(M, N, Hs)
