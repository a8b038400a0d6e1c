"""Shared test helpers: tolerance checks and oracle-side input conversion."""
import numpy as np
import torch

# Floating-point bar for every CUDA output against the fp64 oracle run on the same
# bf16-rounded inputs: relative Frobenius error per tensor and absolute error per element.
REL_FRO_TOL = 1e-2
MAX_ABS_TOL = 3e-2


def f64(t):
    """Exact widening of a (bf16/fp32) tensor to a float64 numpy array."""
    return t.detach().to("cpu").double().numpy()


def i64(t):
    return t.detach().to("cpu").numpy().astype(np.int64)


def errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff)) / denom if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(got, ref, name, rel_tol=REL_FRO_TOL, abs_tol=MAX_ABS_TOL):
    if isinstance(got, torch.Tensor):
        got = f64(got)
    assert got.shape == np.shape(ref), f"{name}: shape {got.shape} vs {np.shape(ref)}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    max_abs, rel = errors(got, ref)
    assert max_abs <= abs_tol and rel <= rel_tol, \
        f"{name}: max abs {max_abs:.3e} (tol {abs_tol}), rel fro {rel:.3e} (tol {rel_tol})"
    return max_abs, rel


class PerExpert:
    """Per-expert fp64 view of an [E, a, b] bf16 tensor that converts on access."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].double().cpu().numpy()

    def __len__(self):
        return self.t.shape[0]
