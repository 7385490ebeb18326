"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before any CUDA call.
(Pointers here are fake addresses; validation never dereferences them.)"""
import ctypes
import os
import re

import pytest

from kimi_k3_attention_gb300 import binding
from kimi_k3_attention_gb300.build import LIB

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attnres.h")

pytestmark = pytest.mark.skipif(not os.path.exists(LIB), reason="libattnres.so not built")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attnres_\w+)\s*\(", src)))


def test_header_declarations_are_exported():
    lib = ctypes.CDLL(LIB)
    names = _declared()
    assert set(names) == set(binding.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version():
    for code in binding.STATUS:
        assert binding.status_string(code)
    assert binding.status_string(12345) == "unknown status"
    assert binding.version() >= 100


M, N, H = 4, 3, 64
R = M * H * 2
BASE = 1 << 32


def _layout():
    """Disjoint fake device regions, 16-byte aligned."""
    off = [0]

    def take(n):
        a = BASE + off[0]
        off[0] += (n + 4095) // 4096 * 4096
        return a
    return dict(prefix=take(R), add=take(R), add2=take(R), bank=take(N * R), w=take(2 * H),
                gamma=take(2 * H), out=take(R), new_prefix=take(R))


def _call(**kw):
    a = _layout()
    a.update({k: v for k, v in kw.items() if k in a})
    shape = dict(M=M, N=N, H=H, eps=1e-6)
    shape.update({k: v for k, v in kw.items() if k in shape})
    return binding.attnres_add_rmsnorm_raw(a["prefix"], a["add"], a["add2"], a["bank"], a["w"],
                                           a["gamma"], shape["eps"], a["out"], a["new_prefix"],
                                           shape["M"], shape["N"], shape["H"])


@pytest.mark.parametrize("kw,code", [
    (dict(prefix=0), -1), (dict(add=0), -1), (dict(bank=0), -1), (dict(w=0), -1),
    (dict(gamma=0), -1), (dict(out=0), -1), (dict(new_prefix=0), -1),
    (dict(N=-1), -2), (dict(N=32), -2), (dict(M=0), -2), (dict(H=12), -2), (dict(H=0), -2),
    (dict(H=16392), -2),
    (dict(eps=0.0), -5), (dict(eps=-1e-6), -5), (dict(eps=float("inf")), -5), (dict(eps=float("nan")), -5),
    (dict(prefix=BASE + 8), -3), (dict(bank=BASE + (1 << 20) + 2), -3), (dict(out=BASE + (9 << 20) + 4), -3),
])
def test_invalid_arguments_rejected(kw, code):
    assert _call(**kw) == code


def test_alias_rules():
    a = _layout()
    # out inside the bank
    assert _call(out=a["bank"] + 16) == -4
    # out equal to new_prefix
    assert _call(out=a["new_prefix"]) == -4
    # out overlapping w
    assert _call(out=a["w"] - 16) == -4
    # new_prefix overlapping add2, or partly overlapping prefix
    assert _call(new_prefix=a["add2"] + 32) == -4
    assert _call(new_prefix=a["prefix"] + 16) == -4
    # new_prefix inside the bank snapshots the call reads
    assert _call(new_prefix=a["bank"] + R) == -4


def test_config_struct_layout():
    c = binding.make_config("cluster", cluster=8, threads=128)
    assert ctypes.sizeof(c) == 32
    assert c.as_dict() == {"variant": 2, "cluster": 8, "threads": 128, "grid_tokens": 0, "pdl": 0,
                           "stages": 0, "prefetch": 0, "tail_tokens": 0}


def test_new_entry_points_validate_on_host():
    a = _layout()
    lib = binding.load()
    vp = ctypes.c_void_p
    # tap: h_out required, must not overlap out
    assert lib.attnres_add_rmsnorm_tap(vp(a["prefix"]), vp(a["add"]), vp(a["add2"]), vp(a["bank"]),
                                       vp(a["w"]), vp(a["gamma"]), 1e-6, vp(a["out"]),
                                       vp(a["new_prefix"]), None, M, N, H, None) == -1
    assert lib.attnres_add_rmsnorm_tap(vp(a["prefix"]), vp(a["add"]), vp(a["add2"]), vp(a["bank"]),
                                       vp(a["w"]), vp(a["gamma"]), 1e-6, vp(a["out"]),
                                       vp(a["new_prefix"]), vp(a["out"] + 32), M, N, H, None) == -4
    # alone: no addends needed, but the usual checks hold
    assert lib.attnres_rmsnorm(vp(a["prefix"]), None, vp(a["w"]), vp(a["gamma"]), 1e-6,
                               vp(a["out"]), M, N, H, None) == -1
    assert lib.attnres_rmsnorm(vp(a["prefix"]), vp(a["bank"]), vp(a["w"]), vp(a["gamma"]), 1e-6,
                               vp(a["bank"] + 64), M, N, H, None) == -4
    assert lib.attnres_rmsnorm(vp(a["prefix"]), vp(a["bank"]), vp(a["w"]), vp(a["gamma"]), 1e-6,
                               vp(a["out"]), M, 32, H, None) == -2
    # N = 0 needs no bank, but N > 0 does
    assert lib.attnres_rmsnorm(vp(a["prefix"]), None, vp(a["w"]), vp(a["gamma"]), 1e-6,
                               vp(a["out"]), M, 1, H, None) == -1
    # tail add
    assert lib.attnres_tail_add(vp(a["prefix"]), None, None, vp(a["new_prefix"]), M, H, None) == -1
    assert lib.attnres_tail_add(vp(a["prefix"]), vp(a["add"]), None, vp(a["new_prefix"]), M, 12, None) == -2
    assert lib.attnres_tail_add(vp(a["prefix"]), vp(a["add"]), None, vp(a["add"] + 16), M, H, None) == -4
    assert lib.attnres_tail_add(vp(a["prefix"] + 4), vp(a["add"]), None, vp(a["new_prefix"]), M, H, None) == -3
    # generic launch: NULL args
    assert lib.attnres_launch(None, None, None) == -1


def _c_layout():
    """sizeof / offsetof of the header's structs, from a C program compiled
    against include/attnres.h."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {"attnres_args": [f for f, _ in binding.Args._fields_],
              "attnres_config": [f for f, _ in binding.Config._fields_]}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "attnres.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'  printf("{st} sizeof %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'  printf("{st} {f} %zu\\n", offsetof({st}, {f}));')
    lines += ["  return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        open(src, "w").write("\n".join(lines) + "\n")
        subprocess.run([cc, "-I", os.path.dirname(HEADER), src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    return {tuple(l.split()[:2]): int(l.split()[2]) for l in out.splitlines()}


@pytest.mark.parametrize("py,c", [(binding.Args, "attnres_args"), (binding.Config, "attnres_config")])
def test_struct_layouts_match_the_header(py, c):
    lay = _c_layout()
    assert ctypes.sizeof(py) == lay[(c, "sizeof")]
    for f, _ in py._fields_:
        assert getattr(py, f).offset == lay[(c, f)], f


def test_fp16_validation_on_host():
    a = _layout()
    lib = binding.load()
    vp = ctypes.c_void_p
    args = [vp(a["prefix"]), vp(a["add"]), vp(a["add2"]), vp(a["bank"]), vp(a["w"]), vp(a["gamma"]),
            1e-6, vp(a["out"]), vp(a["new_prefix"])]
    # FP16 takes the same shapes as BF16
    assert lib.attnres_add_rmsnorm_f16(*args, M, 32, H, None) == -2
    # the usual checks hold for FP16 too
    assert lib.attnres_add_rmsnorm_f16(*args[:7], vp(a["add"]), vp(a["new_prefix"]), M, N, H, None) == -4
    assert lib.attnres_add_rmsnorm_f16(*args, M, N, 12, None) == -2
    # an unknown element type
    x = binding.Args(a["prefix"], a["add"], a["add2"], a["bank"], a["w"], a["gamma"], 1e-6, a["out"],
                     a["new_prefix"], None, M, N, H, 1, 2)
    assert lib.attnres_launch(ctypes.byref(x), None, None) == -9
