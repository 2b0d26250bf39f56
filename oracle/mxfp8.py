"""CPU oracle for the tile-scaled FP8 grouped expert GEMM (forward).

TEST INFRASTRUCTURE ONLY, like moe_oracle: imported by the tests and never by
the library. Plain NumPy, float64 arithmetic; shares no code with the CUDA
path.

Source: xtuner PR "Decouple expert parallelism from FSDP sharding (dp2ep
layout)", "Changes" (the Float8 bullet: per-class padding and tile-wise
scaling) and "Verification" (tile-wise FP8 runs of Qwen3-MoE and GLM-5.2);
the pages name tile-wise FP8 training but give no element format, tile shape,
scale type or rounding.

Reading adopted (the block-scaled FP8 format the GB300 tensor cores take
natively, the OCP Microscaling "MXFP8" format):
* elements are FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
  bits; no infinities; largest finite 448; subnormals down to 2^-9);
* every 32 consecutive elements along the reduction dimension K share one
  power-of-two scale 2^X stored as an 8-bit biased exponent (E8M0, code
  X + 127);
* X = floor(log2(max |v| of the block)) - 8, the largest-magnitude element's
  exponent less E4M3's largest exponent, clamped to [-127, 127]; an all-zero
  block takes X = -127;
* each element is v / 2^X rounded to the nearest E4M3 value, ties to even,
  magnitudes beyond 448 saturating to 448;
* the GEMM multiplies the dequantized values (element * 2^X) exactly and
  sums them (float64 here, fp32 on the GPU).
In the SwiGLU expert the three GEMMs quantize their operands along their own
K: X (rows of the dispatched tokens) and W_gate, W_up along d; H and W_down
along I. H itself is stored in bf16 (as in the bf16 path) and quantized from
that. Parity: pinned by the CPU tests (exhaustive E4M3 decode and rounding
against torch's float8_e4m3fn, closed-form scale rule and round trips, a
hand-worked block, the reduction to the bf16 layer when quantization is
exact).
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import _silu, round_bf16

E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest finite E4M3 value (448 = 1.75 * 2^8)
BLOCK = 32

__all__ = ["e4m3_decode", "e4m3_round", "e4m3_encode", "mx_quantize", "mx_dequantize",
           "grouped_ffn_mxfp8", "E4M3_MAX", "BLOCK"]


def _floor_log2(a):
    """floor(log2(a)) for a > 0, exactly (from the binary exponent); 0 where a == 0."""
    _, e = np.frexp(np.asarray(a, dtype=np.float64))     # a = m * 2^e, m in [0.5, 1)
    return np.where(np.asarray(a) > 0, e - 1, 0).astype(np.int64)


def e4m3_decode(code):
    """Value of each E4M3 code (uint8): sign bit 7, exponent bits 6..3 (bias 7),
    mantissa bits 2..0; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return s * val


def e4m3_round(y):
    """Nearest E4M3 value to each y (float64), ties to even, saturating at 448.
    In the normal range |y| in [2^q, 2^(q+1)), q >= -6, the spacing is 2^(q-3);
    below 2^-6 it is the subnormal spacing 2^-9. Dividing by the spacing is
    exact, so rint (halves to even) picks the correctly rounded multiple."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    q = np.maximum(_floor_log2(a), -6)
    step = np.ldexp(1.0, q - 3)
    r = np.rint(a / step) * step
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(np.where(a > 0, r, 0.0), y)


def e4m3_encode(y):
    """Code of e4m3_round(y) (uint8); -0.0 and +0.0 both give code 0."""
    r = e4m3_round(y)
    a = np.abs(r)
    sign = np.where(r < 0, 0x80, 0)
    sub = a < 2.0 ** -6
    q = _floor_log2(a)
    exp = np.where(sub, 0, q + 7)
    mant = np.where(sub, np.rint(a / 2.0 ** -9), np.rint((a / np.ldexp(1.0, q) - 1.0) * 8))
    code = sign | (exp << 3) | mant.astype(np.int64)
    return np.where(a == 0, 0, code).astype(np.uint8)


def mx_quantize(v, axis: int = -1):
    """Blocks of 32 consecutive elements along ``axis`` (its length a multiple
    of 32). Returns (elements, X): elements as E4M3 values (float64, exactly
    representable) with the block's shared exponent X (int64, one per block,
    the blocked axis shortened 32-fold)."""
    v = np.moveaxis(np.asarray(v, dtype=np.float64), axis, -1)
    n = v.shape[-1]
    if n % BLOCK:
        raise ValueError("the blocked axis must be a multiple of 32")
    b = v.reshape(v.shape[:-1] + (n // BLOCK, BLOCK))
    amax = np.abs(b).max(axis=-1)
    X = np.where(amax > 0, _floor_log2(amax) - E4M3_EMAX, -127).astype(np.int64)
    X = np.clip(X, -127, 127)
    q = e4m3_round(b / np.ldexp(1.0, X)[..., None])
    q = q.reshape(v.shape)
    return np.moveaxis(q, -1, axis), np.moveaxis(X, -1, axis)


def mx_dequantize(q, X, axis: int = -1):
    """element * 2^X, X broadcast over each block of 32 along ``axis``."""
    q = np.moveaxis(np.asarray(q, dtype=np.float64), axis, -1)
    Xm = np.moveaxis(np.asarray(X), axis, -1)
    s = np.repeat(np.ldexp(1.0, Xm.astype(np.int64)), BLOCK, axis=-1)
    return np.moveaxis(q * s, -1, axis)


def _mx(v, axis):
    return mx_dequantize(*mx_quantize(v, axis), axis=axis)


def grouped_ffn_mxfp8(xp, offsets, Wg, Wu, Wd, pre: bool = False):
    """The SwiGLU experts of the grouped FFN with every GEMM on MXFP8 operands:
    per expert e on rows [offsets[e], offsets[e+1]):
    G = mx(X) mx(Wg[e]), U = mx(X) mx(Wu[e]) (X and the weights blocked along d),
    GU = bf16([G | U]), H = bf16(silu(G) * U), Y = bf16(mx(H) mx(Wd[e])) (H and
    W_down blocked along I). Returns y, gu, h (with ``pre``: y, gu, h before
    their own bf16 rounding, Y still from the rounded H)."""
    xp = np.asarray(xp, dtype=np.float64)
    E = len(offsets) - 1
    I = np.asarray(Wg).shape[-1]
    d = np.asarray(Wd).shape[-1]
    n = xp.shape[0]
    y = np.zeros((n, d))
    gu = np.zeros((n, 2 * I))
    h = np.zeros((n, I))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        X = _mx(xp[lo:hi], axis=1)
        G = X @ _mx(Wg[e], axis=0)
        U = X @ _mx(Wu[e], axis=0)
        Hx = _silu(G) * U
        H = round_bf16(Hx)
        Yx = _mx(H, axis=1) @ _mx(Wd[e], axis=0)
        if pre:
            y[lo:hi], gu[lo:hi], h[lo:hi] = Yx, np.concatenate([G, U], axis=1), Hx
        else:
            y[lo:hi], gu[lo:hi], h[lo:hi] = (round_bf16(Yx), round_bf16(np.concatenate([G, U], 1)),
                                             H)
    return y, gu, h
