"""Comparison helpers shared by the parity tests (tolerances of the pages' targets)."""
import numpy as np
import torch

# bf16 inputs, fp32 accumulation: forward and gradient targets
MAX_ABS = 2e-2
REL_FRO = 5e-3
LSE_ABS = 1e-3


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def errors(got, ref):
    g, r = to64(got), to64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    d = g - r
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    den = float(np.linalg.norm(r.ravel()))
    rel = float(np.linalg.norm(d.ravel()) / den) if den > 0 else float(np.linalg.norm(d.ravel()))
    return max_abs, rel


def storage_half_ulp(got):
    """Half an ulp of each element in the output's storage format (0 for fp32/fp64).
    A bf16 output can never be closer to the exact value than this."""
    if isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16:
        g = np.abs(to64(got))
        e = np.floor(np.log2(np.where(g > 0, g, 1.0)))
        ulp = np.where(g > 0, 2.0 ** (e - 7), 2.0 ** -133)
        return 0.5 * ulp
    return 0.0


def assert_close(got, ref, name, max_abs=MAX_ABS, rel_fro=REL_FRO):
    """max-abs: error beyond the output's own storage rounding,
    max(|got - ref| - half_ulp(got)); relative Frobenius against the fp64 oracle."""
    d = np.abs(to64(got) - to64(ref)) - storage_half_ulp(got)
    ma = float(max(np.max(d), 0.0)) if d.size else 0.0
    _, rf = errors(got, ref)
    assert ma <= max_abs and rf <= rel_fro, f"{name}: max_abs={ma:.3e} (<= {max_abs}), rel_fro={rf:.3e} (<= {rel_fro})"
    return ma, rf


def assert_lse(got, ref, name="lse", tol=LSE_ABS):
    g, r = to64(got), to64(ref)
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin), f"{name}: -inf pattern differs"
    assert np.all(g[~fin] == r[~fin]), f"{name}: non-finite values differ"
    if fin.any():
        err = float(np.max(np.abs(g[fin] - r[fin])))
        assert err <= tol, f"{name}: max |d| = {err:.3e} > {tol}"

