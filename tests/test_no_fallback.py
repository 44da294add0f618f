"""The product path has no CPU or PyTorch fallback: every step of the
attention runs in the CUDA library, and a call without the library fails
instead of computing something else.  (CPU tests: no GPU needed.)"""
import ast
import os

import pytest
import torch

import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import _lib, build as _build

PKG = os.path.dirname(os.path.abspath(A.__file__))

# Calls that would compute attention (or part of it) in PyTorch.
_ARITH = {"softmax", "log_softmax", "matmul", "bmm", "baddbmm", "einsum", "exp", "exp2", "tanh",
          "logsumexp", "scaled_dot_product_attention", "mm", "addmm"}


def _py_sources():
    for root, _, files in os.walk(PKG):
        if "_build" in root:
            continue
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(root, f)


def test_package_python_does_no_attention_arithmetic():
    """No `@`, no softmax / matmul / exp style call and no oracle import in the
    package's Python: it only marshals arguments to the C ABI (inputs.py, the
    seeded input generator, only draws random numbers)."""
    for path in _py_sources():
        tree = ast.parse(open(path).read(), path)
        for node in ast.walk(tree):
            assert not (isinstance(node, ast.BinOp) and isinstance(node.op, ast.MatMult)), \
                f"{path}:{node.lineno} uses @"
            if isinstance(node, ast.Call):
                f = node.func
                name = f.attr if isinstance(f, ast.Attribute) else getattr(f, "id", "")
                assert name not in _ARITH, f"{path}:{node.lineno} calls {name}"
            if isinstance(node, (ast.Import, ast.ImportFrom)):
                mods = [a.name for a in node.names] + [getattr(node, "module", None) or ""]
                assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), \
                    f"{path}:{node.lineno} imports the oracle"


def test_call_without_the_library_raises(monkeypatch):
    """With the library neither loaded nor buildable, an entry point raises
    rather than returning a result."""
    def no_build(*args, **kwargs):
        raise RuntimeError("library unavailable")

    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_build, "build", no_build)
    monkeypatch.setattr(_build, "LIB", os.path.join(PKG, "_build", "no_such_library.so"))
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(RuntimeError, match="library unavailable"):
        A.attn_fwd(q, q, q)
    with pytest.raises(RuntimeError, match="library unavailable"):
        A.attn_fwd_varlen(q[0].transpose(0, 1).contiguous(), q[0].transpose(0, 1).contiguous(),
                          q[0].transpose(0, 1).contiguous(),
                          torch.tensor([0, 8], dtype=torch.int32),
                          torch.tensor([0, 8], dtype=torch.int32), 8)
