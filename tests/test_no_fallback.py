"""The product path has no CPU fallback: CPU tensors and a missing library
raise instead of computing anything (no GPU needed)."""
import pytest
import torch

import rmsnorm_backward_gb300 as gbn


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(gbn, "_lib", None)
    monkeypatch.setattr(gbn, "library_path", "/nonexistent/libgbnorm.so")
    with pytest.raises(RuntimeError, match="not built"):
        gbn.lib()


def test_cpu_tensors_are_rejected():
    x = torch.randn(4, 64)
    g = torch.ones(64)
    rstd = torch.ones(4)
    mean = torch.zeros(4)
    with pytest.raises(ValueError, match="CUDA"):
        gbn.rms_fwd(x, g, 1e-6)
    with pytest.raises(ValueError, match="CUDA"):
        gbn.rms_bwd(x, x, g, rstd)
    with pytest.raises(ValueError, match="CUDA"):
        gbn.ln_bwd(x, x, g, mean, rstd)
    with pytest.raises(ValueError):
        gbn.silu_bwd(x, x)
    with pytest.raises(ValueError):
        gbn.gelu_bwd(x, x)


def test_package_does_not_import_the_oracle():
    import ast
    import inspect
    tree = ast.parse(inspect.getsource(gbn))
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            assert all(not a.name.startswith("oracle") for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            assert not (node.module or "").startswith("oracle")
