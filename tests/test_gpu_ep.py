"""Expert parallelism over R ranks on one GPU: every rank's kernels run for
real and the collectives are device copies (LoopbackExchange).

All-to-all EP regroups exactly the rows of each expert, in the same order, as
the single-GPU layer packs them, so its outputs and gradients are compared
bit for bit with the single-GPU layer (MoELayer) on the same inputs, and its
per-rank receive layout with the simulated layout of moe_ep_layout. The
all-gather / reduce-scatter design sums fp32 partials over the ranks, so its
out and dx are compared with the oracle at the bf16 tolerances (and its
expert and router gradients bit for bit with the single-GPU layer). Both are
also compared with the oracle's layer. Cases include a rank that receives no
token."""
import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import ep as EP
from grouped_gemm_moe_gb300 import layer as L
from grouped_gemm_moe_gb300 import workloads as W
from oracle import moe_oracle as O

from _parity import assert_out_close, assert_rms_close, dev, ensure_built, f64, i64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


CASES = [
    W.small_config("ep4", T=1024, d=256, E=16, K=4, I=256, R=4),
    W.small_config("ep2_shared", T=512, d=128, E=8, K=2, I=128, R=2, shared_I=256),
    W.small_config("ep8_skew", T=2048, d=256, E=32, K=4, I=128, R=8, skew=True),
    W.small_config("ep2_idle_rank", T=512, d=128, E=8, K=2, I=256, R=2, seed=3),
    W.small_config("ep4_norenorm", T=512, d=128, E=16, K=3, I=128, R=4, renorm=0),
    W.small_config("ep8_qwen3_shape", T=2048, d=2048, E=128, K=8, I=768, R=8),
    # hidden and intermediate sizes that are multiples of 8 only
    W.small_config("ep2_odd", T=512, d=136, E=8, K=2, I=200, R=2, shared_I=72),
]


def _inputs(cfg):
    inp = W.make_inputs(cfg, with_backward=True)
    if cfg.name == "ep2_idle_rank":
        # rank 1's experts (4..7) are never selected: it receives no token
        inp["logits"][:, cfg.E // 2:] -= 100.0
    return inp


def _single(cfg, inp):
    layer = L.layer_from_config(cfg, inp, dev())
    out = layer.forward(inp["logits"].to(dev()), inp["x"].to(dev())).clone()
    dx = layer.backward(inp["dout"].to(dev())).clone()
    return layer, out, dx


def _chunks(t, R):
    return [c.contiguous() for c in t.to(dev()).chunk(R)]


def _oracle(cfg, inp):
    np_inp = {k: W.to_f64(v) for k, v in inp.items()}
    ref = O.layer_forward(np_inp, cfg.K, cfg.R, cfg.renorm, pre=True)
    rb = O.layer_backward(np_inp, ref, np_inp["dout"], cfg.K, cfg.renorm, pre=True)
    return ref, rb


def _weights(cfg, inp):
    keys = ["w_gate", "w_up", "w_down"] + (["ws_gate", "ws_up", "ws_down"] if cfg.shared_I else [])
    return {k: inp[k].to(dev()).contiguous() for k in keys}


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_all_to_all_ep_matches_single_gpu_layer(cfg):
    inp = _inputs(cfg)
    R, El = cfg.R, cfg.E // cfg.R
    layer, out1, dx1 = _single(cfg, inp)
    w = _weights(cfg, inp)
    ranks = [EP.A2ARank(r, R, cfg.T // R, cfg.d, cfg.E, cfg.K, cfg.I, EP.local_weights(w, r, R),
                        cfg.renorm, dev()) for r in range(R)]
    ex = EP.LoopbackExchange(R)
    outs = EP.a2a_forward(ranks, ex, _chunks(inp["logits"], R), _chunks(inp["x"], R))
    dxs = EP.a2a_backward(ranks, ex, _chunks(inp["dout"], R))
    torch.cuda.synchronize()
    for rk in ranks:
        assert B_status(rk) == 0
    # bit for bit with the single-GPU layer
    assert torch.equal(torch.cat(outs), out1)
    assert torch.equal(torch.cat(dxs), dx1)
    assert torch.equal(torch.cat([rk.dlogits for rk in ranks]), layer.dlogits)
    assert torch.equal(torch.cat([rk.dtopk_w for rk in ranks]), layer.dtopk_w)
    for k in ("dw_gate", "dw_up", "dw_down"):
        assert torch.equal(torch.cat([getattr(rk, k) for rk in ranks]), getattr(layer, k)), k
    if cfg.shared_I:   # the shared expert's weight gradient is the sum over the ranks' tokens
        got = sum(f64(rk.dws_gate) for rk in ranks)
        assert np.allclose(got, f64(layer.dws_gate), rtol=1e-4, atol=1e-6 * np.abs(got).max())
    # each rank's receive layout is its block of the simulated layout
    S = i64(layer.ep_splits)[R * cfg.E:].reshape(R, R)          # S[source][destination]
    glob_reg, off = i64(layer.regroup_index), i64(layer.offsets)
    recv_base = np.concatenate([[0], np.cumsum(S.sum(0))])
    for r, rk in enumerate(ranks):
        assert rk.send_splits == S[r].tolist() and rk.recv_splits == S[:, r].tolist()
        lo, hi = off[r * El], off[(r + 1) * El]
        assert rk.n_recv == hi - lo
        assert np.array_equal(i64(rk.local_offsets), off[r * El:(r + 1) * El + 1] - lo)
        assert np.array_equal(i64(rk.regroup[:rk.n_recv]), glob_reg[lo:hi] - recv_base[r])
    if cfg.name == "ep2_idle_rank":
        assert ranks[1].n_recv == 0 and (f64(ranks[1].dw_gate) == 0).all()
    # and with the oracle's layer
    if cfg.d * cfg.I <= 256 * 256:
        ref, rb = _oracle(cfg, inp)
        assert_out_close(f64(torch.cat(outs)), ref["out_pre"], name="out")
        assert_out_close(f64(torch.cat(dxs)), rb["dx_pre"], name="dx")
        assert_rms_close(f64(torch.cat([rk.dlogits for rk in ranks])), rb["dlogits"], name="dlogits")
        assert_rms_close(f64(torch.cat([rk.dw_down for rk in ranks])), rb["dw_down"], name="dw_down")


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_allgather_reducescatter_ep(cfg):
    inp = _inputs(cfg)
    R = cfg.R
    layer, out1, dx1 = _single(cfg, inp)
    w = _weights(cfg, inp)
    ranks = [EP.AGRSRank(r, R, cfg.T // R, cfg.d, cfg.E, cfg.K, cfg.I, EP.local_weights(w, r, R),
                         cfg.renorm, dev()) for r in range(R)]
    ex = EP.LoopbackExchange(R)
    lg = _chunks(inp["logits"], R)
    outs = EP.agrs_forward(ranks, ex, lg, _chunks(inp["x"], R))
    dxs = EP.agrs_backward(ranks, ex, _chunks(inp["dout"], R), lg)
    torch.cuda.synchronize()
    for rk in ranks:
        assert B_status(rk) == 0
    # the experts' rows and the router are computed exactly as on one GPU
    for k in ("dw_gate", "dw_up", "dw_down"):
        assert torch.equal(torch.cat([getattr(rk, k) for rk in ranks]), getattr(layer, k)), k
    assert torch.equal(torch.cat([rk.dtopk_w for rk in ranks]), layer.dtopk_w)
    assert torch.equal(torch.cat([rk.dlogits for rk in ranks]), layer.dlogits)
    for rk in ranks:
        assert torch.equal(rk.topk_idx, layer.topk_idx)
        assert torch.equal(rk.offsets, layer.offsets)
        n = int(rk.local_offsets[-1])
        lo = int(layer.offsets[rk.e_lo])
        assert torch.equal(rk.y[:n], layer.y[lo:lo + n])
    if cfg.name == "ep2_idle_rank":
        assert int(ranks[1].local_offsets[-1]) == 0
    # out and dx: the fp32 partials are summed over the ranks before the rounding
    ref, rb = _oracle(cfg, inp) if cfg.d * cfg.I <= 256 * 256 else (None, None)
    if ref is not None:
        assert_out_close(f64(torch.cat(outs)), ref["out_pre"], name="out")
        assert_out_close(f64(torch.cat(dxs)), rb["dx_pre"], name="dx")
    else:   # against the single-GPU layer: the same sums in another fp32 order, one rounding
        for got, want, name in ((outs, out1, "out"), (dxs, dx1, "dx")):
            g, wv = f64(torch.cat(got)), f64(want)
            assert (np.abs(g - wv) <= 2 * 2.0 ** -8 * np.abs(wv) + 1e-6).all(), name


def B_status(rk) -> int:
    from grouped_gemm_moe_gb300 import binding as B
    wss = [rk.ws_ffn, rk.ws_bwd] + ([rk.ws_sfwd, rk.ws_sbwd] if rk.shared else [])
    if hasattr(rk, "ws_recv"):
        wss.append(rk.ws_recv)
    for ws in wss:
        s = B.moe_read_device_status(ws)
        if s:
            return s
    return 0
