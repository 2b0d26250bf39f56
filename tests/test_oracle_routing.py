"""Pins of the oracle's bf16 rounding, top-k routing and routing backward.

Each pin comes from something other than the oracle itself: torch's own bf16
conversion, exhaustive enumeration, hand-derived fixtures, torch.topk /
torch.softmax / torch.autograd (independent library code) and finite
differences.
"""
import itertools
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- rounding
def test_round_bf16_matches_torch_conversion():
    g = torch.Generator().manual_seed(1)
    parts = [
        torch.randn(200000, generator=g),
        torch.randn(20000, generator=g) * 1e-38,            # subnormal range
        torch.randn(20000, generator=g) * 3e38,             # near overflow
        torch.randn(20000, generator=g) * 1e6,
    ]
    x = torch.cat(parts).to(torch.float32)
    x = x[torch.isfinite(x)]
    # exact halfway cases: bf16 value + half a bf16 ulp
    base = torch.randn(10000, generator=g).to(torch.bfloat16).to(torch.float32)
    bits = base.view(torch.int32) | 0x8000
    x = torch.cat([x, bits.view(torch.float32), torch.tensor([0.0, -0.0, 1.0, -1.0])])
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(x.to(torch.float64).numpy())
    same = (ref == got) | (np.isnan(ref) & np.isnan(got))
    assert same.all(), (x.numpy()[~same][:5], ref[~same][:5], got[~same][:5])


def test_round_bf16_is_identity_on_bf16_values():
    v = torch.randn(5000).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_bf16(v), v)


# ----------------------------------------------------------------- top-k ids
def _valid_topk(l, ids):
    E = len(l)
    sel = list(ids)
    if len(set(sel)) != len(sel):
        return False
    for j in range(len(sel) - 1):         # slot order: best first, ties to lower id
        a, b = sel[j], sel[j + 1]
        if not (l[a] > l[b] or (l[a] == l[b] and a < b)):
            return False
    for i in sel:
        for u in range(E):
            if u in sel:
                continue
            if not (l[i] > l[u] or (l[i] == l[u] and i < u)):
                return False
    return True


@pytest.mark.parametrize("E", [1, 2, 3, 4, 5])
def test_topk_exhaustive_three_valued(E):
    vals = [-1.0, 0.0, 1.0]
    rows = np.array(list(itertools.product(vals, repeat=E)), dtype=np.float64)
    for K in range(1, E + 1):
        idx, w = O.route_topk(rows, K, renorm=1)
        for r in range(rows.shape[0]):
            ref = sorted(range(E), key=lambda i: (-rows[r, i], i))[:K]
            assert list(idx[r]) == ref
            assert _valid_topk(rows[r], idx[r])
        assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_topk_signed_zero_is_a_tie():
    l = np.array([[-0.0, 0.0, -1.0]])
    idx, _ = O.route_topk(l, 2)
    assert list(idx[0]) == [0, 1]
    l = np.array([[0.0, -0.0, -1.0]])
    idx, _ = O.route_topk(l, 2)
    assert list(idx[0]) == [0, 1]


def test_topk_golden_ties():
    with open(os.path.join(GOLDEN, "topk_ties.txt")) as f:
        lines = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(lines) >= 5
    for ln in lines:
        head, logits, ids, ws = [p.split() for p in ln.split("|")]
        K, renorm = int(head[0]), int(head[1])
        l = np.array([[float(v) for v in logits]])
        idx, w = O.route_topk(l, K, renorm)
        assert list(idx[0]) == [int(v) for v in ids]
        assert np.allclose(w[0], [float(v) for v in ws], rtol=0, atol=1e-15)


def test_topk_all_equal_exact_weights():
    for E, K in [(8, 2), (128, 8), (64, 6), (64, 8)]:
        l = np.full((3, E), 0.25)
        idx, w = O.route_topk(l, K, renorm=1)
        assert (idx == np.arange(K)).all()
        assert (w == 1.0 / K).all() or np.allclose(w, 1.0 / K, rtol=0, atol=1e-16)
        idx, w = O.route_topk(l, K, renorm=0)
        assert np.allclose(w, 1.0 / E, rtol=0, atol=1e-16)


def test_topk_ids_match_torch_topk_on_distinct_logits():
    g = torch.Generator().manual_seed(2)
    l = torch.randn(500, 64, generator=g, dtype=torch.float64)
    for K in (1, 6, 8, 64):
        ref = torch.topk(l, K, dim=1, largest=True, sorted=True).indices.numpy()
        idx, _ = O.route_topk(l.numpy(), K)
        assert np.array_equal(idx, ref)


def test_topk_weights_against_torch_softmax():
    g = torch.Generator().manual_seed(3)
    l = torch.randn(300, 32, generator=g, dtype=torch.float64)
    idx, w0 = O.route_topk(l.numpy(), 5, renorm=0)
    p = torch.softmax(l, dim=1).numpy()
    assert np.allclose(w0, np.take_along_axis(p, idx, 1), rtol=1e-13, atol=0)
    _, w1 = O.route_topk(l.numpy(), 5, renorm=1)
    sel = torch.gather(l, 1, torch.from_numpy(idx.astype(np.int64)))
    assert np.allclose(w1, torch.softmax(sel, dim=1).numpy(), rtol=1e-13, atol=0)
    # ratio invariant w_i / w_j = exp(l_i - l_j)
    li = np.take_along_axis(l.numpy(), idx, 1)
    assert np.allclose(w1[:, 0] / w1[:, 1], np.exp(li[:, 0] - li[:, 1]), rtol=1e-12)
    # full-width renormalised top-k is the plain softmax
    idx, wf = O.route_topk(l.numpy(), 32, renorm=1)
    assert np.allclose(wf, np.take_along_axis(p, idx, 1), rtol=1e-13)


# ----------------------------------------------------------- routing backward
def _torch_route_weights(l, idx, renorm):
    p = torch.softmax(l, dim=1)
    w = torch.gather(p, 1, idx)
    if renorm:
        w = w / w.sum(dim=1, keepdim=True)
    return w


@pytest.mark.parametrize("renorm", [0, 1])
def test_route_backward_against_autograd(renorm):
    g = torch.Generator().manual_seed(4)
    T, E, K = 40, 16, 4
    l = torch.randn(T, E, generator=g, dtype=torch.float64, requires_grad=True)
    dw = torch.randn(T, K, generator=g, dtype=torch.float64)
    idx, w = O.route_topk(l.detach().numpy(), K, renorm)
    wt = _torch_route_weights(l, torch.from_numpy(idx.astype(np.int64)), renorm)
    assert np.allclose(wt.detach().numpy(), w, rtol=1e-13)
    wt.backward(dw)
    got = O.route_topk_backward(l.detach().numpy(), idx, w, dw.numpy(), renorm)
    assert np.allclose(got, l.grad.numpy(), rtol=1e-10, atol=1e-14)
    # softmax shift invariance: each row of dlogits sums to zero
    assert np.allclose(got.sum(axis=1), 0.0, atol=1e-12)
    if renorm:
        mask = np.zeros((T, E), bool)
        np.put_along_axis(mask, idx, True, 1)
        assert (got[~mask] == 0).all()


def test_route_backward_finite_difference():
    rng = np.random.default_rng(5)
    T, E, K = 3, 10, 3
    l = rng.standard_normal((T, E))
    dw = rng.standard_normal((T, K))
    for renorm in (0, 1):
        idx, w = O.route_topk(l, K, renorm)
        dl = O.route_topk_backward(l, idx, w, dw, renorm)
        h = 1e-6
        for t, i in [(0, 0), (1, int(idx[1, 0])), (2, int(idx[2, 2])), (2, 7)]:
            lp = l.copy(); lp[t, i] += h
            lm = l.copy(); lm[t, i] -= h
            # keep the same selection (no tie crossing for these draws)
            ip, wp = O.route_topk(lp, K, renorm)
            im, wm = O.route_topk(lm, K, renorm)
            assert (ip == idx).all() and (im == idx).all()
            fd = ((wp - wm) * dw).sum() / (2 * h)
            assert abs(fd - dl[t, i]) < 1e-7
