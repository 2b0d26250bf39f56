"""GPU parity of the load-balance metrics, loss and gradient against the CPU
oracle (moe_load_balance, moe_load_balance_backward through the C ABI).

Tolerances: load fractions are counts / (T*K) in fp32 (one rounding), so
1e-7 relative; mean probabilities and the loss are fp32 sums of T (or E)
terms, checked at 1e-5 relative; the empty-expert count is exact. The
gradient s * (E/T) * p_i * (f_i - sum_e f_e p_e) subtracts two numbers near
1/E when routing is balanced, so its fp32 error scales with the terms before
the subtraction: max |err| <= 1e-5 * (RMS(g) + RMS(s * (E/T) * p * f))."""
import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import binding as B
from grouped_gemm_moe_gb300 import workloads as W
from oracle import moe_oracle as O

from _parity import ensure_built, f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _case(T, E, K, seed, skew=0.0):
    g = np.random.default_rng(seed)
    l = g.normal(size=(T, E)).astype(np.float32)
    if skew:
        l = l - np.float32(skew) * np.log1p(np.arange(E, dtype=np.float32))
    idx, _ = O.route_topk(l, K, 1)
    counts, _ = O.expert_counts_offsets(idx, E)
    return l, idx, counts.astype(np.int32)


def _assert_grad_close(got, want, l, f, scale, name):
    got = np.asarray(got, dtype=np.float64)
    T, E = l.shape
    terms = scale * (E / T) * O.softmax(l) * f[None, :]
    tol = 1e-5 * (np.sqrt(np.mean(want ** 2)) + np.sqrt(np.mean(terms ** 2)))
    err = np.abs(got - want).max()
    assert np.isfinite(got).all(), name
    assert err <= tol, f"{name}: max|err|={err:.3e} > {tol:.3e}"


def _check_forward(l, idx, counts, E):
    K = idx.shape[1]
    frac, pmean, stats = B.moe_load_balance(to_dev(l, torch.float32), to_dev(counts, torch.int32), K)
    r = O.load_balance(l.astype(np.float64), idx, E)
    np.testing.assert_allclose(f64(frac), r["f"], rtol=1e-7, atol=0)
    np.testing.assert_allclose(f64(pmean), r["P"], rtol=1e-5, atol=1e-9)
    s = f64(stats)
    assert abs(s[0] - r["loss"]) <= 1e-5 * r["loss"]
    assert abs(s[1] - r["max_over_uniform"]) <= 1e-6 * r["max_over_uniform"]
    assert s[2] == r["n_empty"]
    assert abs(s[3] - 1.0) < 1e-5
    return frac, r


@pytest.mark.parametrize("T,E,K,skew", [(64, 8, 2, 0.0), (1000, 128, 8, 0.0), (513, 64, 6, 1.5),
                                        (300, 20, 3, 0.0), (77, 1024, 32, 0.0), (4096, 256, 8, 3.0)])
def test_load_balance_forward_and_backward(T, E, K, skew):
    l, idx, counts = _case(T, E, K, T + E + K, skew)
    frac, r = _check_forward(l, idx, counts, E)
    lt = to_dev(l, torch.float32)
    want = O.load_balance_backward(l.astype(np.float64), r["f"], scale=0.01)
    got = B.moe_load_balance_backward(lt, frac, 0.01)
    _assert_grad_close(f64(got), want, l.astype(np.float64), r["f"], 0.01, "load-balance dlogits")
    # accumulate adds into what is there (a base of the gradient's own size, so the fp32
    # rounding of base + g stays far below the tolerance)
    rms = float(np.sqrt(np.mean(want ** 2)))
    base = torch.randn(T, E, dtype=torch.float32, device=lt.device) * rms
    acc = B.moe_load_balance_backward(lt, frac, 0.01, dlogits=base.clone(), accumulate=True)
    _assert_grad_close(f64(acc) - f64(base), want, l.astype(np.float64), r["f"], 0.01,
                       "accumulated dlogits")


def test_uniform_routing_loss_is_exactly_one():
    T, E, K = 64, 8, 2
    idx = (np.arange(T * K).reshape(T, K) % E).astype(np.int32)
    counts = np.bincount(idx.reshape(-1), minlength=E).astype(np.int32)
    frac, pmean, stats = B.moe_load_balance(torch.zeros(T, E, device="cuda"), to_dev(counts, torch.int32), K)
    s = f64(stats)
    assert s[0] == 1.0 and s[1] == 1.0 and s[2] == 0.0 and s[3] == 1.0
    g = B.moe_load_balance_backward(torch.zeros(T, E, device="cuda"), frac, 1.0)
    assert torch.count_nonzero(g).item() == 0


def test_full_workload_and_determinism():
    cfg = W.CONFIGS["skew"]
    inp = W.make_inputs(cfg, with_backward=False)
    l = inp["logits"].numpy()
    idx, _ = O.route_topk(l, cfg.K, 1)
    counts, _ = O.expert_counts_offsets(idx, cfg.E)
    counts = counts.astype(np.int32)
    frac, r = _check_forward(l, idx, counts, cfg.E)
    lt, ct = to_dev(l, torch.float32), to_dev(counts, torch.int32)
    a = B.moe_load_balance(lt, ct, cfg.K)
    b = B.moe_load_balance(lt, ct, cfg.K)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    g = B.moe_load_balance_backward(lt, frac, 0.5)
    rows = np.random.default_rng(0).choice(cfg.T, size=64, replace=False)
    scale_full = 0.5 * len(rows) / cfg.T     # the oracle on a row subset divides by its own T
    want = O.load_balance_backward(l[rows].astype(np.float64), r["f"], scale=scale_full)
    _assert_grad_close(f64(g)[rows], want, l[rows].astype(np.float64), r["f"], scale_full,
                       "sampled dlogits")
