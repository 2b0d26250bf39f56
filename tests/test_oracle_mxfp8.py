"""Pins of the MXFP8 oracle (oracle/mxfp8.py) on the CPU: exhaustive E4M3
decode and rounding against torch's float8_e4m3fn, the scale rule in closed
form, round trips of exactly representable blocks, hand-worked blocks
(tests/golden/mxfp8_blocks.txt), the blocked axis, and the FP8 expert FFN
reducing to the bf16 oracle when every operand is exactly representable."""
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import mxfp8 as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp8_blocks.txt")


def _torch_e4m3(values):
    return torch.from_numpy(np.asarray(values, dtype=np.float32)).to(
        torch.float8_e4m3fn).float().double().numpy()


def test_decode_every_code_matches_torch():
    codes = np.arange(256)
    ours = M.e4m3_decode(codes)
    ref = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.nanmax(ours) == 448.0 and np.nanmin(np.abs(ours[ours != 0])) == 2.0 ** -9


def test_rounding_matches_torch_on_values_midpoints_and_neighbours():
    vals = np.unique(M.e4m3_decode(np.arange(256)))
    vals = vals[np.isfinite(vals)]
    mids = (vals[1:] + vals[:-1]) / 2
    # fp32-exact test points: the values, the midpoints and their fp32 neighbours
    pts = np.concatenate([vals, mids]).astype(np.float32)
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)),
                          np.nextafter(pts, np.float32(-np.inf))]).astype(np.float64)
    pts = pts[np.abs(pts) < 464.0]           # beyond the 448/480 midpoint torch overflows to NaN
    assert np.array_equal(M.e4m3_round(pts), _torch_e4m3(pts))
    g = np.random.default_rng(0)
    r = (g.standard_normal(200_000) * np.exp(g.standard_normal(200_000) * 3)).astype(np.float32)
    r = r[np.abs(r) < 464.0].astype(np.float64)
    assert np.array_equal(M.e4m3_round(r), _torch_e4m3(r))


def test_saturation_and_encode_roundtrip():
    assert M.e4m3_round(np.array([463.9, 1e6, -1e6]))[0] == 448.0
    assert list(M.e4m3_round(np.array([1e6, -1e6]))) == [448.0, -448.0]
    vals = M.e4m3_decode(np.arange(256))
    fin = np.isfinite(vals)
    codes = M.e4m3_encode(vals[fin])
    assert np.array_equal(M.e4m3_decode(codes), vals[fin])


def test_scale_rule_and_error_bound():
    g = np.random.default_rng(1)
    v = g.standard_normal((64, 256)) * np.exp(g.standard_normal((64, 1)) * 4)
    q, X = M.mx_quantize(v, axis=1)
    b = v.reshape(64, 8, 32)
    amax = np.abs(b).max(-1)
    assert np.array_equal(X, np.floor(np.log2(amax)).astype(np.int64) - 8)
    assert np.abs(q).max() <= 448.0
    # every element is the nearest E4M3 value of v / 2^X: within half a spacing
    scaled = (b / np.ldexp(1.0, X)[..., None]).reshape(64, 256)
    a = np.abs(scaled)
    spacing = np.ldexp(1.0, np.maximum(np.floor(np.log2(np.where(a > 0, a, 1))), -6).astype(int) - 3)
    near = np.abs(q - scaled) <= spacing / 2 + 1e-300
    saturated = (a > 448.0) & (np.abs(q) == 448.0) & (np.sign(q) == np.sign(scaled))
    assert (near | saturated).all() and saturated.any()
    # the block maximum lands in [256, 512): its exponent is E4M3's largest
    top = np.abs(q.reshape(64, 8, 32)).max(-1)
    assert ((top >= 256) & (top <= 448)).all()


def test_exact_blocks_round_trip():
    g = np.random.default_rng(2)
    grid = M.e4m3_decode(np.arange(256))
    grid = grid[np.isfinite(grid)]
    q = g.choice(grid, size=(16, 64))
    q[:, ::32] = 256.0 * np.sign(q[:, ::32] + 0.5)   # each block's max has exponent 8
    X = g.integers(-20, 20, size=(16, 2))
    v = q * np.repeat(np.ldexp(1.0, X), 32, axis=1)
    q2, X2 = M.mx_quantize(v, axis=1)
    assert np.array_equal(X2, X) and np.array_equal(q2, q)
    assert np.array_equal(M.mx_dequantize(q2, X2, axis=1), v)


def _golden():
    blocks, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "block":
            cur = {"v": np.zeros(32), "codes": np.zeros(32, dtype=np.uint8)}
            for item in rest:
                i, val = item.split(":")
                cur["v"][int(i)] = float(val)
            blocks.append(cur)
        elif key == "X":
            cur["X"] = int(rest[0])
        elif key == "codes":
            for item in rest:
                i, c = item.split(":")
                cur["codes"][int(i)] = int(c, 16)
    return blocks


def test_hand_worked_blocks():
    blocks = _golden()
    assert len(blocks) == 3
    for b in blocks:
        q, X = M.mx_quantize(b["v"][None, :], axis=1)
        assert int(X[0, 0]) == b["X"]
        assert np.array_equal(M.e4m3_encode(q[0]), b["codes"])


def test_blocked_axis_is_the_reduction_axis():
    g = np.random.default_rng(3)
    w = g.standard_normal((64, 96))
    q0, X0 = M.mx_quantize(w, axis=0)          # blocks of 32 rows per column
    q1, X1 = M.mx_quantize(w.T, axis=1)
    assert np.array_equal(q0, q1.T) and np.array_equal(X0, X1.T)
    with pytest.raises(ValueError):
        M.mx_quantize(np.ones((3, 40)), axis=1)


def test_fp8_ffn_reduces_to_bf16_ffn_when_quantization_is_exact():
    """Operands whose blocks are already E4M3 values times a power of two pass
    through the quantizer unchanged (and H is made so by construction of Wd
    only through its own blocks), so G and U equal the bf16 oracle's; with an
    H that is exact too, Y does."""
    g = np.random.default_rng(4)
    grid = M.e4m3_decode(np.arange(256))
    grid = grid[np.isfinite(grid) & (np.abs(grid) <= 16)]

    def exact(shape, axis, X):
        q = g.choice(grid, size=shape)
        idx = [slice(None)] * len(shape)
        idx[axis] = slice(0, None, 32)
        q[tuple(idx)] = 256.0                       # each block's max: exponent 8
        return q * 2.0 ** X

    E, d, I = 3, 64, 64
    off = np.array([0, 5, 5, 37])
    xp = exact((37, d), 1, -10)
    Wg = np.stack([exact((d, I), 0, -14) for _ in range(E)])
    Wu = np.stack([exact((d, I), 0, -14) for _ in range(E)])
    Wd = np.stack([exact((I, d), 0, -14) for _ in range(E)])
    y8, gu8, h8 = M.grouped_ffn_mxfp8(xp, off, Wg, Wu, Wd, pre=True)
    yb, gub, hb = O.grouped_ffn(xp, off, Wg, Wu, Wd, pre=True)
    assert np.array_equal(gu8, gub) and np.array_equal(h8, hb)
    # Y differs only through the quantization of the bf16 H: bounded by it
    hq = M.mx_dequantize(*M.mx_quantize(O.round_bf16(hb), axis=1), axis=1)
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        assert np.allclose(y8[lo:hi], hq[lo:hi] @ Wd[e], rtol=1e-12, atol=0)


def test_fp8_ffn_close_to_bf16_ffn():
    g = np.random.default_rng(5)
    E, d, I = 2, 128, 64
    off = np.array([0, 40, 96])
    xp = O.round_bf16(g.standard_normal((96, d)))
    Wg, Wu = (O.round_bf16(g.standard_normal((E, d, I)) * 0.05) for _ in range(2))
    Wd = O.round_bf16(g.standard_normal((E, I, d)) * 0.05)
    y8, _, _ = M.grouped_ffn_mxfp8(xp, off, Wg, Wu, Wd, pre=True)
    yb, _, _ = O.grouped_ffn(xp, off, Wg, Wu, Wd, pre=True)
    rel = np.sqrt(np.mean((y8 - yb) ** 2) / np.mean(yb ** 2))
    assert 1e-3 < rel < 0.1          # FP8's 3 mantissa bits: a few percent, never exact
