"""Shared helpers of the GPU parity tests: building the library, moving seeded
inputs to the device, and the tolerance checks the tests use.

Tolerances (written here once, used by every GPU test):
* integer / index outputs and the dispatch copy: bit-exact;
* fp32 router weights: max |gpu - ref| <= 1e-5 * |ref| (relative, element-wise);
* fp32 weight gradients: max |gpu - ref| <= 2e-2 * RMS(ref) per tensor;
* bf16 results of a sum (y, out, dxp, dx): the same 2e-2 * RMS(ref) bound on the
  error beyond the output's own rounding, max(|gpu - ref| - 2^-8 |ref|, 0),
  where ref is the oracle's value just before that tensor's bf16 rounding (its
  inputs rounded as stored). bf16 keeps 8 significant bits, so rounding alone
  moves an element by up to 2^-8 of its magnitude: 2% of RMS already at 5.1 RMS,
  which a Gaussian tensor of a few million elements exceeds. Against an
  independently rounded reference a single 1-ulp flip at |x| > 2.6 RMS costs
  the same;
* element-wise bf16 intermediates (h, gu): |gpu - ref| <= 2^-8 |ref| +
  1e-3 RMS(ref) against the pre-rounding ref: round-to-nearest moves a value
  by at most half an ulp, 2^-8 of its magnitude, and the slack covers the
  fp32-vs-fp64 accumulation difference before the rounding;
* dy = bf16(w * dout) is rounded once from the exact product: bit-exact;
* fp32 dtopk_w and dlogits fed identical inputs: max |err| <= 1e-3 * RMS(ref).
"""
import numpy as np
import torch

from grouped_gemm_moe_gb300 import build as build_mod

REL_W = 1e-5
RMS_TOL = 2e-2
RMS_TOL_SMALL = 1e-3

_built = False


def ensure_built():
    global _built
    if not _built:
        build_mod.build()
        _built = True


def dev():
    return torch.device("cuda:0")


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def i64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.int64).numpy()


def to_dev(a, dtype) -> torch.Tensor:
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a))
    return a.to(dtype).to(dev()).contiguous()


def assert_rms_close(got, ref, tol=RMS_TOL, name=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert np.isfinite(got).all(), name
    assert err <= tol * rms + 1e-30, f"{name}: max|err|={err:.3e} > {tol}*RMS({rms:.3e})"
    return err / rms if rms else 0.0


def assert_out_close(got, ref_pre, tol=RMS_TOL, name=""):
    """bf16 result of a sum against the oracle's pre-rounding value."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref_pre, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), name
    if not ref.size:
        return 0.0
    rms = np.sqrt(np.mean(ref ** 2))
    excess = np.maximum(np.abs(got - ref) - 2.0 ** -8 * np.abs(ref), 0.0).max()
    assert excess <= tol * rms + 1e-30, (f"{name}: error beyond the bf16 rounding "
                                         f"{excess:.3e} > {tol}*RMS({rms:.3e})")
    return excess / rms if rms else 0.0


def assert_bf16_close(got, ref_pre, name=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref_pre, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * rms
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{name}: {int(bad.sum())} elements outside half an ulp; worst "
                           f"|err|={np.abs(got - ref)[bad].max():.3e}")


def assert_rel_close(got, ref, tol=REL_W, name=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    assert (err <= tol * np.abs(ref) + 1e-30).all(), f"{name}: worst rel err {(err / np.abs(ref)).max():.3e}"
