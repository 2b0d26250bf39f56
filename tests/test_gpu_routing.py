"""GPU parity of router top-k, histogram/offsets/permutation and the simulated
expert-parallel layout against the CPU oracle (bit-exact indices; fp32
weights to 1e-5 relative)."""
import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import binding as B
from grouped_gemm_moe_gb300 import workloads as W
from oracle import moe_oracle as O

from _parity import assert_rel_close, assert_rms_close, dev, ensure_built, f64, i64, to_dev

pytestmark = pytest.mark.gpu

ALL = list(W.CONFIGS)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _logits(cfg):
    g = torch.Generator().manual_seed(cfg.seed)
    l = torch.randn(cfg.T, cfg.E, generator=g, dtype=torch.float32)
    if cfg.skew:
        l = l + W.zipf_bias(cfg.E)
    return l


@pytest.mark.parametrize("name", ALL)
def test_route_topk_workloads(name):
    cfg = W.CONFIGS[name]
    l = _logits(cfg)
    idx, w = B.moe_route_topk(to_dev(l, torch.float32), cfg.K, 1)
    ridx, rw = O.route_topk(l.numpy(), cfg.K, 1)
    assert np.array_equal(i64(idx), ridx)
    assert_rel_close(f64(w), rw, name="topk_w")


@pytest.mark.parametrize("T,E,K,renorm", [(1, 8, 2, 1), (37, 100, 7, 1), (300, 1000, 32, 1),
                                          (64, 33, 32, 0), (513, 64, 6, 0), (1000, 7, 1, 1),
                                          (129, 256, 8, 0), (77, 512, 16, 1)])
def test_route_topk_shapes(T, E, K, renorm):
    g = torch.Generator().manual_seed(T * E + K)
    l = torch.randn(T, E, generator=g) * 3
    idx, w = B.moe_route_topk(to_dev(l, torch.float32), K, renorm)
    ridx, rw = O.route_topk(l.numpy(), K, renorm)
    assert np.array_equal(i64(idx), ridx)
    assert_rel_close(f64(w), rw, name="topk_w")


@pytest.mark.parametrize("E,K", [(8, 2), (128, 8), (64, 6), (40, 5)])
def test_route_topk_ties(E, K):
    # three-valued logits force many exact ties; signed zeros must tie as well
    g = torch.Generator().manual_seed(E)
    l = torch.randint(-1, 2, (512, E), generator=g).to(torch.float32)
    l[::3] = -l[::3]                              # introduces -0.0 entries
    l[5] = 0.0
    idx, w = B.moe_route_topk(to_dev(l, torch.float32), K, 1)
    ridx, rw = O.route_topk(l.numpy(), K, 1)
    assert np.array_equal(i64(idx), ridx)
    assert_rel_close(f64(w), rw, name="topk_w")
    assert (i64(idx)[5] == np.arange(K)).all()


@pytest.mark.parametrize("renorm", [0, 1])
def test_route_topk_backward(renorm):
    T, E, K = 777, 96, 6
    g = torch.Generator().manual_seed(9)
    l = torch.randn(T, E, generator=g)
    ridx, rw = O.route_topk(l.numpy(), K, renorm)
    w32 = torch.from_numpy(rw).to(torch.float32)
    dw = torch.randn(T, K, generator=g)
    dl = B.moe_route_topk_backward(to_dev(l, torch.float32), to_dev(ridx, torch.int32),
                                   to_dev(w32, torch.float32), to_dev(dw, torch.float32), E, renorm)
    ref = O.route_topk_backward(l.numpy(), ridx, w32.double().numpy(), dw.double().numpy(), renorm)
    assert_rms_close(f64(dl), ref, 1e-3, "dlogits")
    if renorm:
        mask = np.ones((T, E), bool)
        np.put_along_axis(mask, ridx.astype(np.int64), False, 1)
        assert (f64(dl)[mask] == 0).all()


def _idx_for(cfg):
    ridx, _ = O.route_topk(_logits(cfg).numpy(), cfg.K, 1)
    return ridx


@pytest.mark.parametrize("name", ALL)
def test_build_permutation_workloads(name):
    cfg = W.CONFIGS[name]
    ridx = _idx_for(cfg)
    counts, offsets, perm, inv = B.moe_build_permutation(to_dev(ridx, torch.int32), cfg.E)
    rc, ro = O.expert_counts_offsets(ridx, cfg.E)
    rp, ri = O.stable_permutation(ridx, cfg.E)
    assert np.array_equal(i64(counts), rc)
    assert np.array_equal(i64(offsets), ro)
    assert np.array_equal(i64(perm), rp)
    assert np.array_equal(i64(inv), ri)


@pytest.mark.parametrize("T,E,K", [(1, 1, 1), (3, 4, 2), (2049, 8, 2), (4096, 1024, 1),
                                   (5000, 3, 3), (1, 1024, 32), (20000, 64, 6)])
def test_build_permutation_shapes(T, E, K):
    rng = np.random.default_rng(T + E)
    ridx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = B.moe_build_permutation(to_dev(ridx, torch.int32), E)
    rc, ro = O.expert_counts_offsets(ridx, E)
    rp, ri = O.stable_permutation(ridx, E)
    assert np.array_equal(i64(counts), rc)
    assert np.array_equal(i64(offsets), ro)
    assert np.array_equal(i64(perm), rp)
    assert np.array_equal(i64(inv), ri)


def test_build_permutation_all_to_one_expert():
    T, E, K = 9000, 16, 1
    ridx = np.full((T, K), 5, dtype=np.int32)
    counts, offsets, perm, inv = B.moe_build_permutation(to_dev(ridx, torch.int32), E)
    assert i64(counts)[5] == T and i64(counts).sum() == T
    assert np.array_equal(i64(perm), np.arange(T))


def _check_ep(ridx, T, E, K, R):
    splits, send, a2a, reg, host = B.moe_ep_layout(to_dev(ridx, torch.int32), E, R)
    torch.cuda.synchronize()
    ref = O.ep_layout(ridx, T, E, K, R)
    s = i64(splits)
    assert np.array_equal(s[:R * E].reshape(R, E), ref["ep_counts"])
    assert np.array_equal(s[R * E:].reshape(R, R), ref["send_splits"])
    assert np.array_equal(host.numpy().astype(np.int64), s)
    assert np.array_equal(i64(send), ref["send_index"])
    assert np.array_equal(i64(a2a), ref["a2a_index"])
    assert np.array_equal(i64(reg), ref["regroup_index"])


@pytest.mark.parametrize("name", ALL)
def test_ep_layout_workloads(name):
    cfg = W.CONFIGS[name]
    _check_ep(_idx_for(cfg), cfg.T, cfg.E, cfg.K, cfg.R)


@pytest.mark.parametrize("T,E,K,R", [(4, 4, 2, 2), (64, 8, 2, 1), (8192, 64, 6, 64),
                                     (6000, 16, 4, 4), (12, 6, 3, 3), (40000, 32, 2, 8)])
def test_ep_layout_shapes(T, E, K, R):
    rng = np.random.default_rng(T * 7 + R)
    ridx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    _check_ep(ridx, T, E, K, R)


def _check_perm_ep(ridx, T, E, K, R):
    out = B.moe_build_permutation_ep(to_dev(ridx, torch.int32), E, R)
    torch.cuda.synchronize()
    counts, offsets, perm, inv, splits, send, a2a, reg, host = out
    rc, ro = O.expert_counts_offsets(ridx, E)
    rp, ri = O.stable_permutation(ridx, E)
    ref = O.ep_layout(ridx, T, E, K, R)
    assert np.array_equal(i64(counts), rc)
    assert np.array_equal(i64(offsets), ro)
    assert np.array_equal(i64(perm), rp)
    assert np.array_equal(i64(inv), ri)
    s = i64(splits)
    assert np.array_equal(s[:R * E].reshape(R, E), ref["ep_counts"])
    assert np.array_equal(s[R * E:].reshape(R, R), ref["send_splits"])
    assert np.array_equal(host.numpy().astype(np.int64), s)
    assert np.array_equal(i64(send), ref["send_index"])
    assert np.array_equal(i64(a2a), ref["a2a_index"])
    assert np.array_equal(i64(reg), ref["regroup_index"])


@pytest.mark.parametrize("name", ALL)
def test_build_permutation_ep_workloads(name):
    """The fused pass gives exactly the outputs of the two separate entry points."""
    cfg = W.CONFIGS[name]
    _check_perm_ep(_idx_for(cfg), cfg.T, cfg.E, cfg.K, cfg.R)


@pytest.mark.parametrize("T,E,K,R", [(4, 4, 2, 2), (64, 8, 2, 1), (8192, 64, 6, 64),
                                     (6000, 16, 4, 4), (12, 6, 3, 3), (3, 1024, 1, 1)])
def test_build_permutation_ep_shapes(T, E, K, R):
    rng = np.random.default_rng(T * 11 + R)
    ridx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    _check_perm_ep(ridx, T, E, K, R)


def _check_route_permute(l, K, R, renorm, ws=None):
    """The fused front against the oracle (route top-k, the permutation and the
    EP layout) and bit for bit against the stand-alone route + permutation."""
    T, E = l.shape
    out = B.moe_route_permute_ep(to_dev(l, torch.float32), K, R, renorm, ws=ws)
    torch.cuda.synchronize()
    idx, w, counts, offsets, perm, inv, splits, send, a2a, reg, host = out
    ridx, rw = O.route_topk(l.numpy(), K, renorm)
    assert np.array_equal(i64(idx), ridx)
    assert_rel_close(f64(w), rw, name="topk_w")
    rc, ro = O.expert_counts_offsets(ridx, E)
    rp, ri = O.stable_permutation(ridx, E)
    ref = O.ep_layout(ridx, T, E, K, R)
    assert np.array_equal(i64(counts), rc)
    assert np.array_equal(i64(offsets), ro)
    assert np.array_equal(i64(perm), rp)
    assert np.array_equal(i64(inv), ri)
    s = i64(splits)
    assert np.array_equal(s[:R * E].reshape(R, E), ref["ep_counts"])
    assert np.array_equal(s[R * E:].reshape(R, R), ref["send_splits"])
    assert np.array_equal(host.numpy().astype(np.int64), s)
    assert np.array_equal(i64(send), ref["send_index"])
    assert np.array_equal(i64(a2a), ref["a2a_index"])
    assert np.array_equal(i64(reg), ref["regroup_index"])
    # the stand-alone kernels give the same bits (weights included)
    sidx, sw = B.moe_route_topk(to_dev(l, torch.float32), K, renorm)
    assert torch.equal(sidx, idx) and torch.equal(sw, w)


@pytest.mark.parametrize("name", ALL)
def test_route_permute_ep_workloads(name):
    cfg = W.CONFIGS[name]
    _check_route_permute(_logits(cfg), cfg.K, cfg.R, cfg.renorm)


@pytest.mark.parametrize("T,E,K,R,renorm", [(4, 4, 2, 2, 1), (64, 8, 2, 1, 0), (8192, 64, 6, 64, 1),
                                            (6000, 16, 4, 4, 1), (12, 6, 3, 3, 0),
                                            (1000, 256, 32, 8, 1), (40000, 32, 2, 8, 0),
                                            (153, 33, 5, 1, 1), (300, 512, 8, 4, 1),
                                            (65536, 128, 8, 8, 1)])
def test_route_permute_ep_shapes(T, E, K, R, renorm):
    """Odd chunk geometries (fewer tokens than SMs, senders of a few tokens,
    chunks of more than 1024 assignments) and E > 256 (the stand-alone path)."""
    g = torch.Generator().manual_seed(T + 13 * E + K)
    _check_route_permute(torch.randn(T, E, generator=g) * 2, K, R, renorm)


def test_route_permute_ep_ties_and_reuse():
    """Three-valued logits (dense ties, signed zeros); the same workspace for
    several calls in a row, with other routings in between."""
    T, E, K, R = 4096, 128, 8, 8
    ws = B.new_workspace(B.workspace_size(B.MOE_OP_ROUTE_PERMUTE_EP, T, E, K, R), dev())
    g = torch.Generator().manual_seed(5)
    for it in range(3):
        l = torch.randint(-1, 2, (T, E), generator=g).to(torch.float32)
        l[::3] = -l[::3]
        if it == 1:
            l = torch.randn(T, E, generator=g)
        _check_route_permute(l, K, R, 1, ws=ws)
    assert B.moe_read_device_status(ws) == 0
