"""GPU parity of the dispatch gather, the weighted combine and their
transposes against the CPU oracle."""
import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import binding as B
from grouped_gemm_moe_gb300 import workloads as W
from oracle import moe_oracle as O

from _parity import assert_out_close, assert_rms_close, ensure_built, f64, i64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _routing(T, E, K, seed, renorm=1):
    g = torch.Generator().manual_seed(seed)
    l = torch.randn(T, E, generator=g)
    idx, w = O.route_topk(l.numpy(), K, renorm)
    perm, inv = O.stable_permutation(idx, E)
    return idx, w.astype(np.float32), perm, inv


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


SHAPES = [(256, 128, 8, 2), (1000, 64, 16, 3), (777, 520, 32, 6), (8192, 2048, 128, 8),
          (1, 8, 4, 4), (3000, 4096, 64, 8),
          # K = 16 and 32 instances of the K-slot kernels; d = 8192 takes the
          # per-row dispatch by perm (rows too long for the bulk-copy ring)
          (100, 136, 64, 16), (50, 8192, 64, 32)]


@pytest.mark.parametrize("T,d,E,K", SHAPES)
def test_dispatch_exact(T, d, E, K):
    _, _, perm, _ = _routing(T, E, K, T + d)
    x = _bf16((T, d), 1)
    xp = B.moe_dispatch(to_dev(x, torch.bfloat16), to_dev(perm, torch.int32), K)
    ref = O.dispatch(x.to(torch.float64).numpy(), perm, K)
    assert np.array_equal(f64(xp), ref)


@pytest.mark.parametrize("T,d,E,K", SHAPES + [(513, 136, 8, 1), (64, 8, 40, 32)])
def test_dispatch_scatter_exact(T, d, E, K):
    """Token-major dispatch through inv_perm: bit-identical to the oracle's gather."""
    _, _, perm, inv = _routing(T, E, K, T + 2 * d)
    x = _bf16((T, d), 4)
    xp = B.moe_dispatch_scatter(to_dev(x, torch.bfloat16), to_dev(inv, torch.int32), K)
    ref = O.dispatch(x.to(torch.float64).numpy(), perm, K)
    assert np.array_equal(f64(xp), ref)


@pytest.mark.parametrize("T,d,E,K", SHAPES)
@pytest.mark.parametrize("shared", [False, True])
def test_combine(T, d, E, K, shared):
    _, w, perm, inv = _routing(T, E, K, T * 3 + d)
    y = _bf16((T * K, d), 2)
    ys = _bf16((T, d), 3) if shared else None
    out = B.moe_combine(to_dev(y, torch.bfloat16), to_dev(w, torch.float32),
                        to_dev(inv, torch.int32), None if ys is None else to_dev(ys, torch.bfloat16))
    ref = O.combine(y.double().numpy(), w.astype(np.float64), inv, K,
                    None if ys is None else ys.double().numpy(), pre=True)
    assert_out_close(f64(out), ref, name="out")


def test_identity_round_trip_is_exact():
    """Dispatch then combine with identity experts returns x exactly when the
    weights are 1/K with K a power of two (all-equal logits)."""
    T, d, E, K = 4096, 256, 16, 4
    l = torch.zeros(T, E)
    idx, w = B.moe_route_topk(to_dev(l, torch.float32), K, 1)
    _, _, perm, inv = B.moe_build_permutation(idx, E)
    x = _bf16((T, d), 5)
    xd = to_dev(x, torch.bfloat16)
    xp = B.moe_dispatch(xd, perm, K)
    out = B.moe_combine(xp, w, inv)
    assert torch.equal(out, xd)


@pytest.mark.parametrize("T,d,E,K", SHAPES)
def test_combine_backward(T, d, E, K):
    _, w, perm, inv = _routing(T, E, K, T * 5 + d)
    y = _bf16((T * K, d), 6)
    dout = _bf16((T, d), 7)
    dy, dw = B.moe_combine_backward(to_dev(dout, torch.bfloat16), to_dev(y, torch.bfloat16),
                                    to_dev(w, torch.float32), to_dev(inv, torch.int32))
    rdy, rdw = O.combine_backward(dout.double().numpy(), y.double().numpy(),
                                  w.astype(np.float64), inv, K)
    assert np.array_equal(f64(dy), rdy), "dy must be the correctly rounded product"
    assert_rms_close(f64(dw), rdw, 1e-3, name="dtopk_w")


@pytest.mark.parametrize("T,d,E,K", SHAPES)
@pytest.mark.parametrize("shared", [False, True])
def test_dispatch_backward(T, d, E, K, shared):
    _, _, perm, inv = _routing(T, E, K, T * 7 + d)
    dxp = _bf16((T * K, d), 8)
    dxs = _bf16((T, d), 9) if shared else None
    dx = B.moe_dispatch_backward(to_dev(dxp, torch.bfloat16), to_dev(inv, torch.int32), T, K,
                                 None if dxs is None else to_dev(dxs, torch.bfloat16))
    ref = O.dispatch_backward(dxp.double().numpy(), inv, K, T,
                              None if dxs is None else dxs.double().numpy(), pre=True)
    assert_out_close(f64(dx), ref, name="dx")


def test_combine_backward_rounding_midpoints():
    """dy = bf16(w * dout) rounded once from the exact product, on inputs where
    the fp32-rounded product lands exactly on a bf16 midpoint: there a second
    rounding of the fp32 product would go the wrong way about half the time."""
    T, d = 2048, 4096
    g = np.random.default_rng(11)
    dout = torch.from_numpy(g.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy(g.uniform(0.05, 1.0, T).astype(np.float32))
    # midpoint cases of this draw (fp32 product's low 16 bits == 0x8000 and inexact)
    prod32 = (dout.float() * w[:, None]).numpy()
    low = prod32.view(np.uint32) & 0xFFFF
    exact = dout.double().numpy() * w.double().numpy()[:, None]
    mid = (low == 0x8000) & (exact != prod32.astype(np.float64))
    assert mid.sum() > 20, "the draw must contain midpoint products"
    inv = np.arange(T, dtype=np.int32)
    y = torch.zeros(T, d, dtype=torch.bfloat16)
    dy, _ = B.moe_combine_backward(to_dev(dout, torch.bfloat16), to_dev(y, torch.bfloat16),
                                   to_dev(w[:, None].contiguous(), torch.float32),
                                   to_dev(inv, torch.int32))
    rdy, _ = O.combine_backward(dout.double().numpy(), y.double().numpy(),
                                w.double().numpy()[:, None], inv, 1)
    got = f64(dy)
    assert np.array_equal(got, rdy), "dy must be the correctly rounded product"
