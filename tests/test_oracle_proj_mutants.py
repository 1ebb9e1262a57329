"""Plausible mistakes planted in copies of the oracle's projection functions (Python source,
re-imported from a temporary module) must be caught by the projection pin."""
import importlib.util
import inspect
import sys

import pytest

import oracle
from _pins import pin_qkv_projection

MUTANTS = [
    ("w_transposed", "_heads(x @ _f64(w), H)", "_heads(x @ _f64(w).T, H)"),
    ("heads_interleaved", "y.reshape(B, N, H, D // H).transpose(0, 2, 1, 3)",
     "y.reshape(B, N, D // H, H).transpose(0, 3, 1, 2)"),
    ("dx_missing_term", "dx += g @ _f64(w).T", "dx = g @ _f64(w).T"),
    ("dw_transposed", "dws.append(xf.T @ g)", "dws.append((xf.T @ g).T)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_projection_pin_catches_mutant(name, old, new, tmp_path, monkeypatch):
    src = inspect.getsource(oracle)
    assert old in src, name
    path = tmp_path / f"oracle_{name}.py"
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"oracle_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    import _pins
    monkeypatch.setattr(_pins, "oracle", mod)
    with pytest.raises(AssertionError):
        pin_qkv_projection(None)
