"""GPU parity of the tcgen05 grouped SwiGLU GEMMs (forward and backward)
against the CPU oracle: every element on small ragged problems, sampled rows
and sampled weight-gradient columns at the workloads' full sizes. Tolerance:
max |err| <= 2e-2 * RMS(reference) per tensor."""
import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import binding as B
from grouped_gemm_moe_gb300 import workloads as W
from oracle import moe_oracle as O

from _parity import assert_bf16_close, assert_out_close, assert_rms_close, ensure_built, f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(*shape, generator=gen) * scale).to(torch.bfloat16)


def _problem(counts, d, I, seed):
    g = torch.Generator().manual_seed(seed)
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    xp = _bf16((M, d), g)
    wg = _bf16((E, d, I), g, 0.02)
    wu = _bf16((E, d, I), g, 0.02)
    wd = _bf16((E, I, d), g, 0.02)
    return off, xp, wg, wu, wd


SMALL = [
    # (counts per expert, d, I)
    ([40, 0, 300, 1, 127, 128, 129, 64], 128, 256),
    ([513, 255, 0, 0, 77], 256, 384),
    ([1000], 512, 128),
    ([63, 65, 200, 1, 0, 319], 384, 512),
    ([0, 0, 0, 5], 256, 256),
    # every width of transposed tail tile (last pair of an expert with 1..128 rows),
    # normal partial tiles (129, 255), exact multiples of 256, and a tail that ends the
    # packed rows (its activation boxes reach past M)
    ([1, 16, 17, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129, 257, 384, 552, 255, 256, 0, 40],
     256, 256),
    # d and I multiples of 8 only: K and N tails inside a 64-column box (the weights'
    # 3-D maps and the half maps of [G | U] and [dG | dU] read zeros past the edge,
    # the stores clip at it); 64 + 64-column gate/up tiles (I % 128 = 8), dW row and
    # column tiles that end inside a box, and dimensions below one box
    ([40, 0, 300, 1, 129], 136, 264),
    ([200, 17, 0, 333], 200, 72),
    ([1, 100, 0, 64, 130], 56, 40),
    ([3, 0, 70, 129], 8, 16),
    ([17, 200], 24, 8),
]


@pytest.mark.parametrize("counts,d,I", SMALL)
def test_grouped_ffn_forward_small(counts, d, I):
    off, xp, wg, wu, wd = _problem(counts, d, I, sum(counts) + d)
    y, h, gu = B.moe_grouped_ffn(to_dev(xp, torch.bfloat16), to_dev(off, torch.int32),
                                 to_dev(wg, torch.bfloat16), to_dev(wu, torch.bfloat16),
                                 to_dev(wd, torch.bfloat16))
    ry, rgu, rh = O.grouped_ffn(xp.double().numpy(), off, wg.double().numpy(),
                                wu.double().numpy(), wd.double().numpy(), pre=True)
    assert_bf16_close(f64(h), rh, name="h")
    assert_bf16_close(f64(gu), rgu, name="gu")
    assert_out_close(f64(y), ry, name="y")


@pytest.mark.parametrize("counts,d,I", SMALL)
def test_grouped_ffn_backward_small(counts, d, I):
    off, xp, wg, wu, wd = _problem(counts, d, I, 3 * sum(counts) + I)
    g = torch.Generator().manual_seed(11)
    M = int(off[-1])
    dy = _bf16((M, d), g, 0.1)
    gu = _bf16((M, 2 * I), g, 1.0)
    h = _bf16((M, I), g, 0.5)
    dxp, dwg, dwu, dwd = B.moe_grouped_ffn_backward(
        to_dev(dy, torch.bfloat16), to_dev(xp, torch.bfloat16), to_dev(gu, torch.bfloat16),
        to_dev(h, torch.bfloat16), to_dev(off, torch.int32), to_dev(wg, torch.bfloat16),
        to_dev(wu, torch.bfloat16), to_dev(wd, torch.bfloat16))
    r = O.grouped_ffn_backward(dy.double().numpy(), xp.double().numpy(), gu.double().numpy(),
                               h.double().numpy(), off, wg.double().numpy(), wu.double().numpy(),
                               wd.double().numpy(), pre=True)
    assert_out_close(f64(dxp), r[0], name="dxp")
    assert_rms_close(f64(dwg), r[1], name="dw_gate")
    assert_rms_close(f64(dwu), r[2], name="dw_up")
    assert_rms_close(f64(dwd), r[3], name="dw_down")
    for e, c in enumerate(counts):
        if c == 0:
            assert (f64(dwg[e]) == 0).all() and (f64(dwd[e]) == 0).all()


def test_shared_expert_as_single_group():
    """E = 1 with offsets {0, T} is the dense always-on expert."""
    T, d, Is = 700, 256, 2 * 384
    g = torch.Generator().manual_seed(5)
    x = _bf16((T, d), g)
    wg, wu = _bf16((1, d, Is), g, 0.02), _bf16((1, d, Is), g, 0.02)
    wd = _bf16((1, Is, d), g, 0.02)
    off = np.array([0, T], np.int32)
    y, h, gu = B.moe_grouped_ffn(to_dev(x, torch.bfloat16), to_dev(off, torch.int32),
                                 to_dev(wg, torch.bfloat16), to_dev(wu, torch.bfloat16),
                                 to_dev(wd, torch.bfloat16), save_gu=False)
    assert gu is None
    ry, _, rh = O.swiglu_expert(x.double().numpy(), wg[0].double().numpy(), wu[0].double().numpy(),
                                wd[0].double().numpy(), pre=True)
    assert_out_close(f64(y), ry, name="y")
    assert_bf16_close(f64(h), rh, name="h")


# ------------------------------------------------------------ full workloads
def _full(name):
    cfg = W.CONFIGS[name]
    inp = W.make_inputs(cfg, with_backward=False)
    idx, _ = O.route_topk(inp["logits"].numpy(), cfg.K, 1)
    counts, off = O.expert_counts_offsets(idx, cfg.E)
    perm, _ = O.stable_permutation(idx, cfg.E)
    return cfg, inp, counts, off.astype(np.int32), perm


def _sample_rows(off, counts, n_per=3, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    nz = np.nonzero(counts)[0]
    pick = set([int(nz[0]), int(nz[-1]), int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])])
    pick |= set(rng.choice(nz, size=min(4, len(nz)), replace=False).tolist())
    for e in sorted(pick):
        lo, hi = int(off[e]), int(off[e + 1])
        cand = {lo, hi - 1, min(lo + 127, hi - 1), min(lo + 128, hi - 1)}
        cand |= set(rng.integers(lo, hi, size=n_per).tolist())
        rows += [(e, p) for p in sorted(cand)]
    return rows


@pytest.mark.parametrize("name", ["qwen3", "dsv2lite", "skew", "drafter"])
def test_grouped_ffn_forward_full_sampled(name):
    cfg, inp, counts, off, perm = _full(name)
    K = cfg.K
    dxd = to_dev(inp["x"], torch.bfloat16)
    xp = B.moe_dispatch(dxd, to_dev(perm, torch.int32), K)
    wg, wu, wd = (to_dev(inp[k], torch.bfloat16) for k in ("w_gate", "w_up", "w_down"))
    y, h, gu = B.moe_grouped_ffn(xp, to_dev(off, torch.int32), wg, wu, wd)
    torch.cuda.synchronize()
    rows = _sample_rows(off, counts)
    ps = torch.tensor([p for _, p in rows])
    yg, hg, gug = f64(y[ps.to(y.device)]), f64(h[ps.to(h.device)]), f64(gu[ps.to(gu.device)])
    ry, rh, rgu = [], [], []
    x64 = inp["x"]
    for (e, p) in rows:
        X = x64[int(perm[p]) // K].double().numpy()[None]
        a, b, c = O.swiglu_expert(X, inp["w_gate"][e].double().numpy(),
                                  inp["w_up"][e].double().numpy(), inp["w_down"][e].double().numpy(),
                                  pre=True)
        ry.append(a[0]); rgu.append(b[0]); rh.append(c[0])
    assert_out_close(yg, np.array(ry), name="y")
    assert_bf16_close(hg, np.array(rh), name="h")
    assert_bf16_close(gug, np.array(rgu), name="gu")


@pytest.mark.parametrize("name", ["qwen3", "dsv2lite", "skew", "drafter"])
def test_grouped_ffn_backward_full_sampled(name):
    cfg, inp, counts, off, perm = _full(name)
    K, d, I, E = cfg.K, cfg.d, cfg.I, cfg.E
    M = cfg.TK
    g = torch.Generator().manual_seed(21)
    dy = _bf16((M, d), g, 0.1)
    gu = _bf16((M, 2 * I), g, 1.0)
    h = _bf16((M, I), g, 0.5)
    xd = to_dev(inp["x"], torch.bfloat16)
    xp = B.moe_dispatch(xd, to_dev(perm, torch.int32), K)
    wg, wu, wd = (to_dev(inp[k], torch.bfloat16) for k in ("w_gate", "w_up", "w_down"))
    dxp, dwg, dwu, dwd = B.moe_grouped_ffn_backward(
        to_dev(dy, torch.bfloat16), xp, to_dev(gu, torch.bfloat16), to_dev(h, torch.bfloat16),
        to_dev(off, torch.int32), wg, wu, wd)
    torch.cuda.synchronize()
    x = inp["x"]
    # sampled rows of dxp
    rows = _sample_rows(off, counts, n_per=2, seed=1)
    ps = torch.tensor([p for _, p in rows])
    got = f64(dxp[ps.to(dxp.device)])
    ref = []
    for (e, p) in rows:
        X = x[int(perm[p]) // K].double().numpy()[None]
        r = O.swiglu_expert_backward(dy[p:p + 1].double().numpy(), X, gu[p:p + 1].double().numpy(),
                                     h[p:p + 1].double().numpy(), inp["w_gate"][e].double().numpy(),
                                     inp["w_up"][e].double().numpy(), inp["w_down"][e].double().numpy(),
                                     pre=True)
        ref.append(r[0][0])
    assert_out_close(got, np.array(ref), name="dxp rows")
    # sampled columns of the weight gradients, restricted-column sub-problems of the oracle
    rng = np.random.default_rng(2)
    nz = np.nonzero(counts)[0]
    experts = sorted(set([int(nz[0]), int(nz[-1]), int(nz[np.argmax(counts[nz])])]))
    cols = np.sort(rng.choice(I, size=4, replace=False))
    for e in experts:
        lo, hi = int(off[e]), int(off[e + 1])
        X = x[torch.from_numpy(perm[lo:hi] // K)].double().numpy()
        GU = gu[lo:hi].double().numpy()
        sub_gu = np.concatenate([GU[:, cols], GU[:, I + cols]], axis=1)
        r = O.swiglu_expert_backward(dy[lo:hi].double().numpy(), X, sub_gu,
                                     h[lo:hi, cols].double().numpy(),
                                     inp["w_gate"][e][:, cols].double().numpy(),
                                     inp["w_up"][e][:, cols].double().numpy(),
                                     inp["w_down"][e][cols, :].double().numpy())
        ci = torch.from_numpy(cols).to(dwg.device)
        assert_rms_close(f64(dwg[e][:, ci]), r[1], name=f"dw_gate[{e}]")
        assert_rms_close(f64(dwu[e][:, ci]), r[2], name=f"dw_up[{e}]")
        assert_rms_close(f64(dwd[e][ci, :]), r[3], name=f"dw_down[{e}]")
    empty = np.nonzero(counts == 0)[0]
    for e in empty[:4]:
        assert float(dwg[int(e)].abs().max()) == 0.0 and float(dwd[int(e)].abs().max()) == 0.0


@pytest.mark.parametrize("E", [600, 1024])
def test_grouped_ffn_many_experts(E):
    """Expert counts past the deep rings' shared-memory budget (the GEMMs fall back
    to their shallower rings; the weight gradients use five stages above 440
    experts), up to the largest supported E: sparse ragged sizes, many experts
    empty, every row compared, forward and backward."""
    rng = np.random.default_rng(E)
    counts = np.where(rng.random(E) < 0.4, 0, rng.integers(1, 40, E))
    d, I = 128, 128
    off, xp, wg, wu, wd = _problem(counts.tolist(), d, I, E)
    args = [to_dev(t, torch.bfloat16) for t in (xp,)] + [to_dev(off, torch.int32)] + \
        [to_dev(t, torch.bfloat16) for t in (wg, wu, wd)]
    y, h, gu = B.moe_grouped_ffn(*args)
    ry, rgu, rh = O.grouped_ffn(xp.double().numpy(), off, wg.double().numpy(), wu.double().numpy(),
                                wd.double().numpy(), pre=True)
    assert_bf16_close(f64(h), rh, name="h")
    assert_bf16_close(f64(gu), rgu, name="gu")
    assert_out_close(f64(y), ry, name="y")
    g = torch.Generator().manual_seed(E + 1)
    M = int(off[-1])
    dy = _bf16((M, d), g, 0.1)
    gu_in = _bf16((M, 2 * I), g, 1.0)
    h_in = _bf16((M, I), g, 0.5)
    dxp, dwg, dwu, dwd = B.moe_grouped_ffn_backward(
        to_dev(dy, torch.bfloat16), args[0], to_dev(gu_in, torch.bfloat16),
        to_dev(h_in, torch.bfloat16), args[1], args[2], args[3], args[4])
    r = O.grouped_ffn_backward(dy.double().numpy(), xp.double().numpy(), gu_in.double().numpy(),
                               h_in.double().numpy(), off, wg.double().numpy(), wu.double().numpy(),
                               wd.double().numpy(), pre=True)
    assert_out_close(f64(dxp), r[0], name="dxp")
    assert_rms_close(f64(dwg), r[1], name="dw_gate")
    assert_rms_close(f64(dwu), r[2], name="dw_up")
    assert_rms_close(f64(dwd), r[3], name="dw_down")
    empty = counts == 0
    assert (f64(dwg)[empty] == 0).all() and (f64(dwd)[empty] == 0).all()


def test_grouped_ffn_no_rows():
    """A batch that routes no row to any expert (M = 0): the forward writes
    nothing and returns, the backward writes zero weight gradients everywhere
    (over whatever the output buffers held)."""
    E, d, I = 4, 128, 128
    off, xp, wg, wu, wd = _problem([0] * E, d, I, 3)
    dv = [to_dev(t, torch.bfloat16) for t in (xp, wg, wu, wd)]
    offd = to_dev(off, torch.int32)
    y, h, gu = B.moe_grouped_ffn(dv[0], offd, dv[1], dv[2], dv[3])
    assert y.shape[0] == 0 and h.shape[0] == 0
    empty_rows = torch.empty(0, d, dtype=torch.bfloat16, device=dv[0].device)
    out = (torch.empty(0, d, dtype=torch.bfloat16, device=dv[0].device),
           torch.full((E, d, I), 7.0, device=dv[0].device),
           torch.full((E, d, I), 7.0, device=dv[0].device),
           torch.full((E, I, d), 7.0, device=dv[0].device))
    dxp, dwg, dwu, dwd = B.moe_grouped_ffn_backward(
        empty_rows, dv[0], torch.empty(0, 2 * I, dtype=torch.bfloat16, device=dv[0].device),
        torch.empty(0, I, dtype=torch.bfloat16, device=dv[0].device), offd, dv[1], dv[2], dv[3],
        out=out)
    torch.cuda.synchronize()
    assert dxp.shape[0] == 0
    assert (dwg == 0).all() and (dwu == 0).all() and (dwd == 0).all()


@pytest.mark.parametrize("counts,d,I", [SMALL[0], SMALL[-1]])
def test_grouped_ffn_backward_split_matches_whole(counts, d, I):
    """The data part then the weight part (with another kernel in between on the
    same stream) give bit-identical results to the single backward call."""
    off, xp, wg, wu, wd = _problem(counts, d, I, 5 * sum(counts) + I)
    g = torch.Generator().manual_seed(13)
    M = int(off[-1])
    dy, gu, h = _bf16((M, d), g, 0.1), _bf16((M, 2 * I), g, 1.0), _bf16((M, I), g, 0.5)
    dv = {k: to_dev(t, torch.bfloat16) for k, t in
          (("dy", dy), ("xp", xp), ("gu", gu), ("h", h), ("wg", wg), ("wu", wu), ("wd", wd))}
    offd = to_dev(off, torch.int32)
    whole = B.moe_grouped_ffn_backward(dv["dy"], dv["xp"], dv["gu"], dv["h"], offd, dv["wg"],
                                       dv["wu"], dv["wd"])
    E = len(counts)
    ws = B.new_workspace(B.workspace_size(B.MOE_OP_GROUPED_FFN_BACKWARD, M, E, 1, 1, d, I),
                         dv["xp"].device)
    dxp = B.moe_grouped_ffn_backward_data(dv["dy"], dv["xp"], dv["gu"], dv["h"], offd, dv["wg"],
                                          dv["wu"], dv["wd"], ws=ws)
    between = B.moe_grouped_ffn(dv["xp"], offd, dv["wg"], dv["wu"], dv["wd"])   # other work
    dws = B.moe_grouped_ffn_backward_weights(dv["dy"], dv["xp"], dv["h"], offd, E, I, ws=ws)
    torch.cuda.synchronize()
    del between
    assert torch.equal(dxp, whole[0])
    for got, want in zip(dws, whole[1:]):
        assert torch.equal(got, want)


def test_grouped_ffn_backward_weights_without_data_part_reports_check():
    """The weight part on a workspace no data part has filled (or filled for
    other offsets) writes nothing and reports MOE_ERR_DEVICE_CHECK; after a
    matching data part it runs normally."""
    counts, d, I = SMALL[0]
    off, xp, wg, wu, wd = _problem(counts, d, I, 7 * sum(counts) + I)
    g = torch.Generator().manual_seed(17)
    M = int(off[-1])
    dy, gu, h = _bf16((M, d), g, 0.1), _bf16((M, 2 * I), g, 1.0), _bf16((M, I), g, 0.5)
    dv = {k: to_dev(t, torch.bfloat16) for k, t in
          (("dy", dy), ("xp", xp), ("gu", gu), ("h", h), ("wg", wg), ("wu", wu), ("wd", wd))}
    offd = to_dev(off, torch.int32)
    E = len(counts)
    dev_ = dv["xp"].device
    ws = B.new_workspace(B.workspace_size(B.MOE_OP_GROUPED_FFN_BACKWARD, M, E, 1, 1, d, I), dev_)
    sentinel = lambda *s: torch.full(s, 7.0, device=dev_)  # noqa: E731
    out = (sentinel(E, d, I), sentinel(E, d, I), sentinel(E, I, d))
    B.moe_grouped_ffn_backward_weights(dv["dy"], dv["xp"], dv["h"], offd, E, I, ws=ws, out=out)
    assert B.moe_read_device_status(ws) == B.MOE_ERR_DEVICE_CHECK
    assert all((t == 7.0).all() for t in out)
    # a data part for another offsets tensor (same values) does not vouch for this one
    off_other = offd.clone()
    B.moe_grouped_ffn_backward_data(dv["dy"], dv["xp"], dv["gu"], dv["h"], off_other, dv["wg"],
                                    dv["wu"], dv["wd"], ws=ws)
    B.moe_grouped_ffn_backward_weights(dv["dy"], dv["xp"], dv["h"], offd, E, I, ws=ws, out=out)
    assert B.moe_read_device_status(ws) == B.MOE_ERR_DEVICE_CHECK
    assert all((t == 7.0).all() for t in out)
    # the matching pair runs and agrees with the single call
    whole = B.moe_grouped_ffn_backward(dv["dy"], dv["xp"], dv["gu"], dv["h"], offd, dv["wg"],
                                       dv["wu"], dv["wd"])
    B.moe_grouped_ffn_backward_data(dv["dy"], dv["xp"], dv["gu"], dv["h"], offd, dv["wg"],
                                    dv["wu"], dv["wd"], ws=ws)
    B.moe_grouped_ffn_backward_weights(dv["dy"], dv["xp"], dv["h"], offd, E, I, ws=ws, out=out)
    assert B.moe_read_device_status(ws) == B.MOE_OK
    for got, want in zip(out, whole[1:]):
        assert torch.equal(got, want)
