"""The product path and the oracle stay apart: importing the package loads no
oracle module, and no file of the package, the kernels or the shared input
generators names the oracle."""
import os
import pathlib
import subprocess
import sys

ROOT = pathlib.Path(__file__).resolve().parents[1]


def test_package_import_loads_no_oracle():
    code = ("import sys, causal_gqa_attention_rmsnorm_gb300 as tb; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300,
                         check=True).stdout.strip().splitlines()[-1]
    assert out == "False"


def test_product_sources_do_not_reference_the_oracle():
    roots = [ROOT / "causal_gqa_attention_rmsnorm_gb300", ROOT / "workloads", ROOT / "include"]
    hits = []
    for r in roots:
        for p in r.rglob("*"):
            if p.suffix in (".py", ".cu", ".cuh", ".h", ".c", ".cpp") and "__pycache__" not in p.parts:
                text = p.read_text(errors="ignore")
                if "import oracle" in text or "from oracle" in text:
                    hits.append(str(p.relative_to(ROOT)))
    assert hits == []


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import pytest
    from causal_gqa_attention_rmsnorm_gb300 import binding
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libtb.so"))
    monkeypatch.setattr(binding, "_lib", None)
    cfg = binding.BlockConfig(64, 4, 2, 16, 176, 16, 1e4, 1e-6, binding.TB_F32)
    with pytest.raises(RuntimeError, match="missing"):
        binding.tb_workspace_bytes(cfg, 1, 16, 0)
