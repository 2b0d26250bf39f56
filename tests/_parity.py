"""Shared helpers of the GPU parity tests: building the library, moving seeded
inputs to the device, and the tolerance checks the tests use.

Tolerances (written here once, used by every GPU test):
* integer / index outputs and the dispatch copy: bit-exact;
* fp32 router weights: max |gpu - ref| <= 1e-5 * |ref| (relative, element-wise);
* fp32 weight gradients: max |gpu - ref| <= 2e-2 * RMS(ref) per tensor;
* bf16 results (y, out, dxp, dx, and the element-wise intermediates h, gu):
  the GPU value is a bf16 rounding of its own fp32 sum, so it may sit up to
  half a bf16 ulp away from that sum. The bound therefore applies to the error
  beyond half an ulp *of the stored GPU value itself*,
  max(|gpu - ref| - ulp(gpu)/2, 0), where ref is the oracle's value just before
  that tensor's bf16 rounding (its inputs rounded as stored) and
  ulp(g) = 2^(floor(log2|g|) - 7) (8 significant bits). For y, out, dxp and dx
  that excess must stay within 2e-2 * RMS(ref) (the stated bf16 bound); for h and gu,
  which are compared element by element, within 1e-3 * RMS(ref) (the fp32 vs
  fp64 accumulation difference before the rounding). Half an ulp of the stored
  value is the largest move a correctly rounded result can make (at a binade
  edge the true bound is half the smaller binade's ulp, which this covers), so
  a value one full ulp off still counts against the budget;
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


def half_ulp_bf16(got) -> np.ndarray:
    """Half a bf16 ulp of each (bf16-exact) value: 2^(floor(log2|g|) - 8); 0 at 0."""
    g = np.abs(np.asarray(got, dtype=np.float64))
    _, e = np.frexp(g)                  # g = m * 2^e with m in [0.5, 1): floor(log2 g) = e - 1
    hu = np.ldexp(1.0, e - 9)
    return np.where(g > 0, hu, 0.0)


def rounding_excess(got, ref_pre) -> np.ndarray:
    """|got - ref| beyond half an ulp of the stored bf16 value got (>= 0)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref_pre, dtype=np.float64)
    return np.maximum(np.abs(got - ref) - half_ulp_bf16(got), 0.0)


def assert_out_close(got, ref_pre, tol=RMS_TOL, name=""):
    """bf16 result of a sum against the oracle's pre-rounding value: the error
    beyond half an ulp of the GPU's stored value within tol * RMS(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref_pre, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), name
    if not ref.size:
        return 0.0
    rms = np.sqrt(np.mean(ref ** 2))
    excess = rounding_excess(got, ref).max()
    assert excess <= tol * rms + 1e-30, (f"{name}: error beyond half an ulp of the stored value "
                                         f"{excess:.3e} > {tol}*RMS({rms:.3e})")
    return excess / rms if rms else 0.0


def assert_bf16_close(got, ref_pre, name=""):
    """Element-wise bf16 intermediate: |gpu - ref| <= ulp(gpu)/2 + 1e-3 * RMS(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref_pre, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), name
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    bad = rounding_excess(got, ref) > RMS_TOL_SMALL * rms
    assert not bad.any(), (f"{name}: {int(bad.sum())} elements beyond half an ulp; worst "
                           f"|err|={np.abs(got - ref)[bad].max():.3e}")


def assert_rel_close(got, ref, tol=REL_W, name=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    assert (err <= tol * np.abs(ref) + 1e-30).all(), f"{name}: worst rel err {(err / np.abs(ref)).max():.3e}"
