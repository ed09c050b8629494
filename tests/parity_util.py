"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (stated for decode attention outputs):
  bf16 inputs/outputs: max |gpu - oracle| <= 1e-2 and ||gpu - oracle|| / ||oracle|| <= 5e-3
  fp32 inputs/outputs: max |gpu - oracle| <= 1e-5 and relative L2 <= 1e-6
The bf16 output grid is coarser than 1e-2 above |x| = 4 (half an ulp there
is 2^-6), so there the element bar is faithful rounding: the output must be
one of the two bf16 values adjacent to the exact result, |gpu - oracle| <
ulp(oracle).  That is the accuracy the method's own arithmetic guarantees:
the weights p are rounded to bf16 before P.V ("FlashMLA на Huawei Ascend",
online softmax), up to 2^-9 relative, i.e. up to half an output ulp before
the output's own rounding.  The relative-L2 bound is unchanged.
Append and gather are byte copies and compare byte for byte.
"""
import numpy as np
import torch

TOL = {torch.bfloat16: (1e-2, 5e-3), torch.float32: (1e-5, 1e-6)}


def bf16_ulp(x):
    """Spacing of the bf16 values around x (8 significant bits)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - 7)


def element_bound(ref, dtype):
    """Per-element bound on |gpu - oracle| (see the module docstring) and the
    mask of elements whose bound is strict (faithful rounding: err < ulp)."""
    max_abs, _ = TOL[dtype]
    bound = np.full_like(ref, max_abs)
    strict = np.zeros(ref.shape, bool)
    if dtype == torch.bfloat16:
        strict = np.abs(ref) >= 4.0
        bound[strict] = bf16_ulp(ref[strict])
    return bound, strict


def violations(err, ref, dtype):
    """Elements whose error breaks the element bound."""
    bound, strict = element_bound(ref, dtype)
    return (err > bound) | (strict & (err >= bound)), bound


def assert_attention_close(gpu, ref, dtype, what=""):
    """gpu: torch tensor (any device, dtype), ref: float64 numpy array."""
    g = gpu.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    _, rel_l2 = TOL[dtype]
    err = np.abs(g - ref)
    bad, bound = violations(err, ref, dtype)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: error {err[i]:.3e} exceeds the bound {bound[i]:.3e} at {i} "
                             f"(oracle {ref[i]:.6g}, gpu {g[i]:.6g}; max abs err {err.max():.3e})")
    nref = np.linalg.norm(ref)
    if nref > 0:
        rel = np.linalg.norm(g - ref) / nref
        assert rel <= rel_l2, f"{what}: relative L2 {rel:.3e} > {rel_l2}"
    else:
        assert np.all(g == 0), f"{what}: expected all zeros"


def assert_lse_close(gpu_lse, ref_lse, what=""):
    """Log-sum-exp rows: -inf exactly where the oracle has -inf, else within
    1e-4 absolute (fp32 accumulation of fp32 scores)."""
    g = gpu_lse.detach().double().cpu().numpy()
    ref = np.asarray(ref_lse, dtype=np.float64)
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), ninf), f"{what}: -inf pattern differs"
    if (~ninf).any():
        d = np.abs(g[~ninf] - ref[~ninf])
        assert d.max() <= 1e-4 * max(1.0, np.abs(ref[~ninf]).max()), f"{what}: lse err {d.max():.3e}"


def host(t):
    return t.detach().cpu()
