"""The product path has no CPU fallback and does not touch the oracle (no GPU
needed): importing the package and its binding loads neither the oracle nor
any module of it, and a missing shared library is an error, not a detour."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_package_import_does_not_load_the_oracle():
    code = ("import sys; import kimi_k3_attention_gb300, kimi_k3_attention_gb300.binding, "
            "kimi_k3_attention_gb300.build, kimi_k3_attention_gb300.workloads; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       check=True)
    assert r.stdout.strip() == "False"


def test_package_sources_do_not_reference_the_oracle():
    pkg = os.path.join(ROOT, "kimi_k3_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_missing_library_is_an_error(tmp_path):
    from kimi_k3_attention_gb300 import binding
    with pytest.raises(RuntimeError):
        binding.load(str(tmp_path / "libattnres.so"))
