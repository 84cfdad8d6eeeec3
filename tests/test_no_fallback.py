"""The product path has no CPU fallback (CPU only).

Every compute entry point of the binding refuses CPU tensors before any
work; a missing library is an error, not a silent substitute; and no module
of the package imports the oracle (only the tests, smoke() and the
benchmark's CPU legs may)."""
import ast
import os

import pytest
import torch

import linear_recurrence_ssm_gb300 as lrs
from linear_recurrence_ssm_gb300 import _build

import workloads

PKG = os.path.dirname(lrs.__file__)


def _diag():
    return workloads.diag_inputs(1, 8, 4, 16, "f32", seed=1)


def _ssd():
    return workloads.ssd_inputs(1, 8, 2, 16, 32, "f32", seed=1)


@pytest.mark.parametrize("call", [
    lambda: lrs.ssm_scan_fwd(**_diag()),
    lambda: lrs.ssm_scan_fwd_bf16(**workloads.diag_inputs(1, 8, 4, 16, "bf16", seed=1)),
    lambda: lrs.ssd_chunk_scan_fwd(**_ssd()),
    lambda: lrs.ssm_scan_bwd(**_diag(), dy=torch.zeros(1, 8, 4)),
    lambda: lrs.ssd_chunk_scan_bwd(**_ssd(), dy=torch.zeros(1, 8, 2, 16)),
])
def test_cpu_tensors_are_refused(call):
    with pytest.raises(ValueError, match="CUDA tensors"):
        call()


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(_build, "needs_build", lambda: False)
    monkeypatch.setattr(lrs, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        lrs.library()


def test_package_never_imports_the_oracle():
    for root, _, files in os.walk(PKG):
        for f in files:
            if not f.endswith(".py"):
                continue
            tree = ast.parse(open(os.path.join(root, f)).read())
            for node in ast.walk(tree):
                names = []
                if isinstance(node, ast.Import):
                    names = [a.name for a in node.names]
                elif isinstance(node, ast.ImportFrom):
                    names = [node.module or ""]
                assert not any(n.split(".")[0] == "oracle" for n in names), (f, names)
