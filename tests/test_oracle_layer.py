"""Pins of the oracle's dispatch, grouped SwiGLU experts, combine and the whole
layer's forward and backward.

Independent references: a per-token torch implementation of the MoE layer
(out[t] = sum_j w_j * MLP_{e_j}(x_t)), torch matmul + F.silu for the dense
E=1 case, torch.autograd in float64 for the backward, algebraic invariants
(identity experts, linearity, expert relabelling), and a hand-worked
two-token example in closed form (tests/golden/swiglu_layer_example.txt).
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from grouped_gemm_moe_gb300 import workloads as W
from oracle import moe_oracle as O


def _np_inputs(cfg, **kw):
    inp = W.make_inputs(cfg, **kw)
    return {k: W.to_f64(v) for k, v in inp.items()}


def _torch_moe_per_token(inp, K, renorm, shared=True):
    """Reference MoE layer written per token with torch ops (fp64, no rounding)."""
    l = torch.from_numpy(inp["logits"])
    x = torch.from_numpy(inp["x"])
    Wg, Wu, Wd = (torch.from_numpy(inp[k]) for k in ("w_gate", "w_up", "w_down"))
    top = torch.topk(l, K, dim=1)
    p = torch.softmax(l, dim=1)
    w = torch.gather(p, 1, top.indices)
    if renorm:
        w = w / w.sum(1, keepdim=True)
    out = torch.zeros_like(x)
    for t in range(x.shape[0]):
        for j in range(K):
            e = int(top.indices[t, j])
            hdn = F.silu(x[t] @ Wg[e]) * (x[t] @ Wu[e])
            out[t] += w[t, j] * (hdn @ Wd[e])
    if shared and "ws_gate" in inp:
        xs = x @ torch.from_numpy(inp["ws_gate"])
        us = x @ torch.from_numpy(inp["ws_up"])
        out += (F.silu(xs) * us) @ torch.from_numpy(inp["ws_down"])
    return out.numpy()


@pytest.mark.parametrize("shared_I", [0, 64])
@pytest.mark.parametrize("renorm", [0, 1])
def test_layer_forward_matches_per_token_torch(shared_I, renorm):
    cfg = W.small_config(T=48, d=32, E=8, K=3, I=48, R=2, shared_I=shared_I, renorm=renorm)
    inp = _np_inputs(cfg)
    res = O.layer_forward(inp, cfg.K, cfg.R, renorm, exact=True)
    ref = _torch_moe_per_token(inp, cfg.K, renorm)
    assert np.allclose(res["out"], ref, rtol=1e-10, atol=1e-12)


def test_layer_forward_rounded_close_to_exact():
    cfg = W.small_config(T=64, d=64, E=8, K=2, I=64, R=2)
    inp = _np_inputs(cfg)
    a = O.layer_forward(inp, cfg.K, cfg.R, 1, exact=False)["out"]
    b = O.layer_forward(inp, cfg.K, cfg.R, 1, exact=True)["out"]
    rms = np.sqrt((b ** 2).mean())
    assert np.abs(a - b).max() < 2e-2 * rms
    assert np.array_equal(O.round_bf16(a), a)


def test_dense_single_expert_against_torch():
    g = torch.Generator().manual_seed(11)
    M, d, I = 37, 64, 96
    X = torch.randn(M, d, generator=g, dtype=torch.float64)
    Wg = torch.randn(1, d, I, generator=g, dtype=torch.float64) * 0.1
    Wu = torch.randn(1, d, I, generator=g, dtype=torch.float64) * 0.1
    Wd = torch.randn(1, I, d, generator=g, dtype=torch.float64) * 0.1
    y, gu, h = O.grouped_ffn(X.numpy(), [0, M], Wg.numpy(), Wu.numpy(), Wd.numpy(), exact=True)
    G, U = X @ Wg[0], X @ Wu[0]
    ref_h = F.silu(G) * U
    assert np.allclose(h, ref_h.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(y, (ref_h @ Wd[0]).numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(gu, torch.cat([G, U], 1).numpy(), rtol=1e-12, atol=1e-14)
    # rounded mode: same as rounding torch's fp32 values at the same points
    Xb = X.to(torch.bfloat16).to(torch.float32)
    Wgb, Wub, Wdb = (w.to(torch.bfloat16).to(torch.float32) for w in (Wg, Wu, Wd))
    y2, gu2, h2 = O.grouped_ffn(Xb.double().numpy(), [0, M], Wgb.double().numpy(),
                                Wub.double().numpy(), Wdb.double().numpy())
    G32, U32 = Xb @ Wgb[0], Xb @ Wub[0]
    h32 = (F.silu(G32) * U32).to(torch.bfloat16).float()
    assert np.abs(h2 - h32.double().numpy()).max() <= 2 ** -7 * np.abs(h32.numpy()).max()


def test_empty_experts_and_grouping():
    rng = np.random.default_rng(3)
    d, I, E = 16, 24, 5
    counts = [3, 0, 4, 0, 2]
    off = np.concatenate([[0], np.cumsum(counts)])
    xp = rng.standard_normal((off[-1], d))
    Wg, Wu = rng.standard_normal((E, d, I)), rng.standard_normal((E, d, I))
    Wd = rng.standard_normal((E, I, d))
    y, gu, h = O.grouped_ffn(xp, off, Wg, Wu, Wd, exact=True)
    for e in range(E):
        for r in range(off[e], off[e + 1]):          # row-wise restatement
            ref = (F.silu(torch.from_numpy(xp[r] @ Wg[e])) * torch.from_numpy(xp[r] @ Wu[e]))
            assert np.allclose(y[r], ref.numpy() @ Wd[e], rtol=1e-12)
    dy = rng.standard_normal(y.shape)
    dxp, dWg, dWu, dWd = O.grouped_ffn_backward(dy, xp, gu, h, off, Wg, Wu, Wd, exact=True)
    for e in (1, 3):
        assert (dWg[e] == 0).all() and (dWu[e] == 0).all() and (dWd[e] == 0).all()


def test_linearity_in_w_down():
    rng = np.random.default_rng(4)
    xp = rng.standard_normal((10, 8))
    off = [0, 4, 10]
    Wg, Wu = rng.standard_normal((2, 8, 12)), rng.standard_normal((2, 8, 12))
    A, B = rng.standard_normal((2, 12, 8)), rng.standard_normal((2, 12, 8))
    ya = O.grouped_ffn(xp, off, Wg, Wu, A, exact=True)[0]
    yb = O.grouped_ffn(xp, off, Wg, Wu, B, exact=True)[0]
    yab = O.grouped_ffn(xp, off, Wg, Wu, 2.0 * A - B, exact=True)[0]
    assert np.allclose(yab, 2 * ya - yb, rtol=1e-11, atol=1e-11)


def test_expert_relabelling_invariance():
    cfg = W.small_config(T=40, d=16, E=8, K=2, I=16, R=2)
    inp = _np_inputs(cfg)
    out = O.layer_forward(inp, 2, 2, 1, exact=True)["out"]
    sig = np.random.default_rng(5).permutation(8)
    inp2 = dict(inp)
    inp2["logits"] = inp["logits"][:, sig]
    for k in ("w_gate", "w_up", "w_down"):
        inp2[k] = inp[k][sig]
    out2 = O.layer_forward(inp2, 2, 2, 1, exact=True)["out"]
    assert np.allclose(out, out2, rtol=1e-12, atol=1e-12)


def test_identity_experts_round_trip():
    """Dispatch then combine with y := xp and renormalised weights returns x."""
    cfg = W.small_config(T=128, d=64, E=8, K=2, I=16, R=2)
    inp = _np_inputs(cfg)
    K = cfg.K
    idx, w = O.route_topk(inp["logits"], K, 1)
    perm, inv = O.stable_permutation(idx, cfg.E)
    xp = O.dispatch(inp["x"], perm, K)
    assert np.array_equal(xp, inp["x"][perm // K])
    out = O.combine(xp, w, inv, K)
    x = inp["x"]
    ulp = np.ldexp(1.0, np.frexp(np.abs(x))[1] - 8)
    assert (np.abs(out - x) <= ulp).all()
    # all-equal logits and K a power of two: w = 1/K exactly, the round trip is exact
    for K in (1, 2, 4, 8):
        l = np.zeros((cfg.T, cfg.E))
        idx, w = O.route_topk(l, K, 1)
        perm, inv = O.stable_permutation(idx, cfg.E)
        out = O.combine(O.dispatch(x, perm, K), w, inv, K)
        assert np.array_equal(out, x)


def test_dispatch_backward_is_transpose_of_dispatch():
    rng = np.random.default_rng(6)
    T, E, K, d = 30, 6, 3, 8
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    perm, inv = O.stable_permutation(idx, E)
    x = rng.standard_normal((T, d))
    g = rng.standard_normal((T * K, d))
    # <dispatch(x), g> == <x, dispatch^T(g)>
    lhs = (O.dispatch(x, perm, K) * g).sum()
    rhs = (x * O.dispatch_backward(g, inv, K, T, exact=True)).sum()
    assert np.isclose(lhs, rhs, rtol=1e-12)


# ------------------------------------------------------------ full backward
def _torch_layer(inp, K, renorm):
    """Layer forward in torch autograd (fp64), packing via index_select / index_add."""
    req = {}
    for k, v in inp.items():
        req[k] = torch.from_numpy(v.copy()).requires_grad_(k != "dout")
    l, x = req["logits"], req["x"]
    T, E = l.shape
    top = torch.topk(l.detach(), K, dim=1).indices
    p = torch.softmax(l, dim=1)
    w = torch.gather(p, 1, top)
    if renorm:
        w = w / w.sum(1, keepdim=True)
    flat = top.reshape(-1)
    order = torch.argsort(flat, stable=True)
    xp = x.index_select(0, order // K)
    y = torch.zeros(T * K, x.shape[1], dtype=x.dtype)
    rows = []
    for e in range(E):
        sel = (flat[order] == e).nonzero().reshape(-1)
        if sel.numel() == 0:
            continue
        X = xp[sel]
        hdn = F.silu(X @ req["w_gate"][e]) * (X @ req["w_up"][e])
        rows.append((sel, hdn @ req["w_down"][e]))
    y = torch.zeros_like(xp).index_put(tuple([torch.cat([s for s, _ in rows])]),
                                        torch.cat([v for _, v in rows]))
    ya = torch.zeros_like(y).index_copy(0, order, y)          # back to token-major
    out = (w.reshape(T * K, 1) * ya).reshape(T, K, -1).sum(1)
    if "ws_gate" in req:
        out = out + (F.silu(x @ req["ws_gate"]) * (x @ req["ws_up"])) @ req["ws_down"]
    out.backward(req["dout"])
    return out.detach().numpy(), {k: v.grad.numpy() for k, v in req.items()
                                  if v.grad is not None}


@pytest.mark.parametrize("shared_I,renorm", [(0, 1), (32, 1), (0, 0), (32, 0)])
def test_layer_backward_against_autograd(shared_I, renorm):
    cfg = W.small_config(T=24, d=16, E=8, K=3, I=24, R=2, shared_I=shared_I, renorm=renorm)
    inp = _np_inputs(cfg)
    fwd = O.layer_forward(inp, cfg.K, cfg.R, renorm, exact=True)
    bwd = O.layer_backward(inp, fwd, inp["dout"], cfg.K, renorm, exact=True)
    out, grads = _torch_layer(inp, cfg.K, renorm)
    assert np.allclose(fwd["out"], out, rtol=1e-10, atol=1e-13)
    assert np.allclose(bwd["dx"], grads["x"], rtol=1e-9, atol=1e-12)
    assert np.allclose(bwd["dlogits"], grads["logits"], rtol=1e-9, atol=1e-12)
    assert np.allclose(bwd["dw_gate"], grads["w_gate"], rtol=1e-9, atol=1e-12)
    assert np.allclose(bwd["dw_up"], grads["w_up"], rtol=1e-9, atol=1e-12)
    assert np.allclose(bwd["dw_down"], grads["w_down"], rtol=1e-9, atol=1e-12)
    if shared_I:
        assert np.allclose(bwd["dws_gate"], grads["ws_gate"], rtol=1e-9, atol=1e-12)
        assert np.allclose(bwd["dws_up"], grads["ws_up"], rtol=1e-9, atol=1e-12)
        assert np.allclose(bwd["dws_down"], grads["ws_down"], rtol=1e-9, atol=1e-12)


def test_backward_finite_difference_on_x():
    cfg = W.small_config(T=6, d=8, E=4, K=2, I=8, R=2)
    inp = _np_inputs(cfg)
    fwd = O.layer_forward(inp, 2, 2, 1, exact=True)
    dout = inp["dout"]
    bwd = O.layer_backward(inp, fwd, dout, 2, 1, exact=True)
    h = 1e-6
    for (t, c) in [(0, 0), (3, 5), (5, 7)]:
        xp_, xm_ = dict(inp), dict(inp)
        xp_["x"] = inp["x"].copy(); xp_["x"][t, c] += h
        xm_["x"] = inp["x"].copy(); xm_["x"][t, c] -= h
        fp = (O.layer_forward(xp_, 2, 2, 1, exact=True)["out"] * dout).sum()
        fm = (O.layer_forward(xm_, 2, 2, 1, exact=True)["out"] * dout).sum()
        assert abs((fp - fm) / (2 * h) - bwd["dx"][t, c]) < 1e-6


def test_workload_shapes_and_skew():
    c = W.CONFIGS
    assert (c["qwen3"].T, c["qwen3"].d, c["qwen3"].E, c["qwen3"].K, c["qwen3"].I) == \
        (8192, 2048, 128, 8, 768)
    assert c["dsv2lite"].shared_I == 2816 and c["drafter"].R == 4
    # the skewed workload: hottest expert above 10x the mean, several experts empty
    cfg = c["skew"]
    g = torch.Generator().manual_seed(0)
    logits = torch.randn(cfg.T, cfg.E, generator=g) + W.zipf_bias(cfg.E)
    idx, _ = O.route_topk(logits.numpy()[:, :], cfg.K, 1)
    counts, _ = O.expert_counts_offsets(idx, cfg.E)
    mean = cfg.T * cfg.K / cfg.E
    assert counts.max() > 10 * mean
    assert (counts == 0).sum() >= 5


def test_pre_rounding_outputs_round_to_the_stored_values():
    """``pre=True`` gives each stored bf16 output just before its rounding:
    rounding it reproduces the stored value, and it is the exact function of
    the (rounded) stored inputs."""
    cfg = W.small_config(T=64, d=64, E=8, K=2, I=64, R=2, shared_I=64)
    inp = _np_inputs(cfg)
    f = O.layer_forward(inp, cfg.K, cfg.R, 1, pre=True)
    for k in ("y", "gu", "h", "out"):
        assert np.array_equal(O.round_bf16(f[k + "_pre"]), f[k]), k
    b = O.layer_backward(inp, f, inp["dout"], cfg.K, 1, pre=True)
    for k in ("dxp", "dx"):
        assert np.array_equal(O.round_bf16(b[k + "_pre"]), b[k]), k
    # y_pre = H_stored @ Wd exactly, segment by segment
    off = f["offsets"]
    for e in range(cfg.E):
        lo, hi = int(off[e]), int(off[e + 1])
        assert np.allclose(f["y_pre"][lo:hi], f["h"][lo:hi] @ inp["w_down"][e], rtol=1e-13, atol=0)


GOLDEN_LAYER = os.path.join(os.path.dirname(__file__), "golden", "swiglu_layer_example.txt")


def _golden_layer():
    """The fixture's 'let' names, evaluated in order, and its expected arrays."""
    env = {"exp": math.exp, "log": math.log}
    want = {}
    for ln in open(GOLDEN_LAYER):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        if ln.startswith("let "):
            k, e = ln[4:].split("=", 1)
            env[k.strip()] = eval(e, {"__builtins__": {}}, env)
        else:
            k, e = ln.split("=", 1)
            want[k.strip()] = np.array(eval(e, {"__builtins__": {}}, env), dtype=np.float64)
    return want


def test_layer_hand_worked_example():
    """tests/golden/swiglu_layer_example.txt: two tokens, two experts with I = 1,
    K = 2, worked by hand in closed form (sigmoid(1), sigmoid(2)) — routing with a
    tie, renormalised weights, the SwiGLU expert and its backward, the combine,
    the router gradient and the per-expert weight gradients; exact arithmetic."""
    want = _golden_layer()
    inp = {"logits": np.array([[0.0, math.log(3.0)], [0.0, 0.0]]),
           "x": np.array([[1.0, 2.0], [0.0, 1.0]]),
           "w_gate": np.array([[[1.0], [0.0]], [[0.0], [1.0]]]),
           "w_up": np.array([[[0.0], [1.0]], [[1.0], [0.0]]]),
           "w_down": np.array([[[3.0, -1.0]], [[1.0, 1.0]]])}
    ref = O.layer_forward(inp, 2, 2, 1, exact=True)
    rb = O.layer_backward(inp, ref, np.array([[1.0, 0.0], [0.0, 1.0]]), 2, 1, exact=True)
    got = {"topk_idx": ref["topk_idx"], "topk_w": ref["topk_w"], "out": ref["out"],
           "dx": rb["dx"], "dtopk_w": rb["dtopk_w"], "dlogits": rb["dlogits"],
           "dw_gate": rb["dw_gate"], "dw_up": rb["dw_up"], "dw_down": rb["dw_down"]}
    assert set(want) == set(got)
    for k, w in want.items():
        g = np.asarray(got[k], dtype=np.float64)
        assert g.shape == w.shape, k
        assert np.allclose(g, w, rtol=0, atol=1e-14), k
