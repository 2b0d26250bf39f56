"""The MXFP8 grouped expert GEMM (forward) against the MXFP8 oracle
(oracle/mxfp8.py): the quantizers bit for bit (every E4M3 value and every
UE8M0 scale, read back from the documented scale-atom layout), and the expert
FFN's h, [G|U] and y element by element on ragged expert segments."""
import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import binding as B
from oracle import moe_oracle as O
from oracle import mxfp8 as MX

from _parity import assert_bf16_close, assert_out_close, dev, ensure_built, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _atom_byte(atom, r, j):
    return atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (j % 4)


def _bf16(shape, g, scale):
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


def _row_tiles(off):
    """First scale tile of each expert: twice the pairs of 128-row m-tiles before it."""
    n = np.diff(off)
    pairs = ((n + 127) // 128 + 1) // 2
    return np.concatenate([[0], 2 * np.cumsum(pairs)])


def _gpu_row_scales(sf, off, K):
    """[M, K/32] scale codes read from the expert-ordered atom layout."""
    sf = sf.cpu().numpy()
    tiles = _row_tiles(off)
    M = int(off[-1])
    out = np.zeros((M, K // 32), dtype=np.int64)
    for e in range(len(off) - 1):
        for r in range(off[e], off[e + 1]):
            loc = r - off[e]
            tile = tiles[e] + loc // 128
            for j in range(K // 32):
                out[r, j] = sf[_atom_byte(tile * (K // 128) + j // 4, loc % 128, j)]
    return out


ROW_CASES = [([40, 0, 300, 1, 127, 128, 129, 64], 256), ([0, 0, 5], 128), ([1000], 512),
             ([63, 65, 200, 1, 0, 319], 384)]


@pytest.mark.parametrize("counts,K", ROW_CASES)
def test_quantize_rows_bit_exact(counts, K):
    g = torch.Generator().manual_seed(sum(counts) + K)
    off = _offsets(counts)
    M = int(off[-1])
    x = _bf16((M, K), g, 1.0)
    x[:, :32] *= 1e-40                     # bf16 subnormals: the scale clamps at 2^-127
    if M > 3:
        x[3, 64:96] = 0                    # an all-zero block
        x[2, 0] = 3.0e38                   # a block near bf16's largest finite
    q, sf = B.moe_mxfp8_quantize_rows(x.to(dev()), torch.from_numpy(off).to(torch.int32).to(dev()))
    torch.cuda.synchronize()
    ref_q, ref_X = MX.mx_quantize(W_f64(x), axis=1)
    got = MX.e4m3_decode(q.cpu().numpy())
    assert np.array_equal(got, ref_q)
    assert np.array_equal(_gpu_row_scales(sf, off, K), ref_X + 127)


def W_f64(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("E,K,N,pair", [(2, 128, 128, False), (3, 256, 384, True),
                                        (1, 512, 256, True), (2, 384, 256, False)])
def test_quantize_weights_bit_exact(E, K, N, pair):
    g = torch.Generator().manual_seed(E * K + N)
    wa = _bf16((E, K, N), g, 0.02)
    wb = _bf16((E, K, N), g, 0.02) if pair else None
    wa[0, :32, 5] = 0                      # an all-zero block
    q, sf = B.moe_mxfp8_quantize_weights(wa.to(dev()), wb.to(dev()) if pair else None)
    torch.cuda.synchronize()
    Nq = 2 * N if pair else N
    got = MX.e4m3_decode(q.cpu().numpy())           # [E, Nq, K]
    sfn = sf.cpu().numpy()
    for e in range(E):
        qa, Xa = MX.mx_quantize(W_f64(wa[e]), axis=0)          # [K, N], [K/32, N]
        if pair:
            qb, Xb = MX.mx_quantize(W_f64(wb[e]), axis=0)
        for n in range(Nq):
            if pair:
                src_b = (n // 128) % 2 == 1
                col = (n // 256) * 128 + n % 128
                rq, rX = (qb, Xb) if src_b else (qa, Xa)
            else:
                col, rq, rX = n, qa, Xa
            assert np.array_equal(got[e, n], rq[:, col]), (e, n)
            atoms = (e * (Nq // 128) + n // 128) * (K // 128)
            codes = [sfn[_atom_byte(atoms + j // 4, n % 128, j)] for j in range(K // 32)]
            assert np.array_equal(np.array(codes), rX[:, col] + 127), (e, n)


FFN_CASES = [
    ([40, 0, 300, 1, 127, 128, 129, 64], 128, 256),
    ([513, 255, 0, 0, 77], 256, 384),
    ([1000], 512, 128),
    ([63, 65, 200, 1, 0, 319], 384, 512),
    ([0, 0, 0, 5], 256, 256),
]


def _ffn_problem(counts, d, I, seed):
    g = torch.Generator().manual_seed(seed)
    E = len(counts)
    off = _offsets(counts)
    M = int(off[-1])
    xp = _bf16((M, d), g, 1.0)
    wg, wu = _bf16((E, d, I), g, 0.02), _bf16((E, d, I), g, 0.02)
    wd = _bf16((E, I, d), g, 0.02)
    return off, xp, wg, wu, wd


def _run_fp8(off, xp, wg, wu, wd):
    D = dev()
    wgu = B.moe_mxfp8_quantize_weights(wg.to(D), wu.to(D))
    wdq = B.moe_mxfp8_quantize_weights(wd.to(D))
    offd = torch.from_numpy(off).to(torch.int32).to(D)
    y, h, gu = B.moe_grouped_ffn_fp8(xp.to(D), offd, wgu, wdq)
    torch.cuda.synchronize()
    return y, h, gu, offd


@pytest.mark.parametrize("counts,d,I", FFN_CASES)
def test_grouped_ffn_fp8_matches_oracle(counts, d, I):
    off, xp, wg, wu, wd = _ffn_problem(counts, d, I, 11 * sum(counts) + d + I)
    y, h, gu, _ = _run_fp8(off, xp, wg, wu, wd)
    ref_y, ref_gu, ref_h = MX.grouped_ffn_mxfp8(W_f64(xp), off, W_f64(wg), W_f64(wu), W_f64(wd),
                                                pre=True)
    assert_bf16_close(f64(h), ref_h, name="h")
    assert_bf16_close(f64(gu), ref_gu, name="gu")
    assert_out_close(f64(y), ref_y, name="y")


def test_grouped_ffn_fp8_without_saved_gu():
    """save_gu=False: the gate/up epilogue stores H (and its E4M3 copy) only; y and
    h are the same as with [G | U] saved."""
    counts = [300, 0, 129, 640, 1, 257]
    d, I = 256, 384
    off, xp, wg, wu, wd = _ffn_problem(counts, d, I, 77)
    y, h, _, offd = _run_fp8(off, xp, wg, wu, wd)
    D = dev()
    wgu = B.moe_mxfp8_quantize_weights(wg.to(D), wu.to(D))
    wdq = B.moe_mxfp8_quantize_weights(wd.to(D))
    y2, h2, gu2 = B.moe_grouped_ffn_fp8(xp.to(D), offd, wgu, wdq, save_gu=False)
    torch.cuda.synchronize()
    assert gu2 is None
    assert torch.equal(y2, y) and torch.equal(h2, h)


def test_grouped_ffn_fp8_many_experts_and_against_bf16():
    """64 experts of ~512 rows at d=2048, I=768 (the qwen3 workload's expert
    shape): the oracle on every row; and the FP8 result stays within FP8's
    precision of the bf16 GEMM on the same inputs."""
    g = np.random.default_rng(21)
    counts = list(np.maximum(0, np.round(512 + g.standard_normal(64) * 21)).astype(int))
    counts[5] = 0
    off, xp, wg, wu, wd = _ffn_problem(counts, 2048, 768, 12)
    y, h, gu, offd = _run_fp8(off, xp, wg, wu, wd)
    ref_y, ref_gu, ref_h = MX.grouped_ffn_mxfp8(W_f64(xp), off, W_f64(wg), W_f64(wu), W_f64(wd),
                                                pre=True)
    assert_bf16_close(f64(h), ref_h, name="h")
    assert_out_close(f64(y), ref_y, name="y")
    D = dev()
    yb, _, _ = B.moe_grouped_ffn(xp.to(D), offd, wg.to(D), wu.to(D), wd.to(D))
    torch.cuda.synchronize()
    a, b = f64(y), f64(yb)
    rel = np.sqrt(np.mean((a - b) ** 2) / np.mean(b ** 2))
    assert rel < 0.1, rel
