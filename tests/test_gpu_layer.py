"""End-to-end GPU layer (forward + backward as a chain of library calls)
against the oracle's layer, and the single device-to-host copy per layer."""
import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import layer as L
from grouped_gemm_moe_gb300 import workloads as W
from oracle import moe_oracle as O

from _parity import (assert_bf16_close, assert_out_close, assert_rel_close, assert_rms_close, dev,
                     ensure_built, f64, i64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


CASES = [
    W.CONFIGS["tiny"],
    W.small_config("ep4", T=512, d=256, E=16, K=4, I=256, R=4),
    W.small_config("shared", T=384, d=128, E=8, K=2, I=128, R=2, shared_I=256),
    W.small_config("skewed", T=1024, d=128, E=32, K=4, I=128, R=8, skew=True),
    W.small_config("norenorm", T=256, d=128, E=8, K=3, I=128, R=2, renorm=0),
]


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_layer_forward_backward(cfg):
    inp = W.make_inputs(cfg, with_backward=True)
    np_inp = {k: W.to_f64(v) for k, v in inp.items()}
    layer = L.layer_from_config(cfg, inp, dev())
    logits = inp["logits"].to(dev())
    x = inp["x"].to(dev())
    dout = inp["dout"].to(dev())
    out = layer.forward(logits, x)
    dx = layer.backward(dout)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    ref = O.layer_forward(np_inp, cfg.K, cfg.R, cfg.renorm, pre=True)
    assert np.array_equal(i64(layer.topk_idx), ref["topk_idx"])
    assert_rel_close(f64(layer.topk_w), ref["topk_w"], name="topk_w")
    assert np.array_equal(i64(layer.counts), ref["counts"])
    assert np.array_equal(i64(layer.offsets), ref["offsets"])
    assert np.array_equal(i64(layer.perm), ref["perm"])
    assert np.array_equal(i64(layer.inv_perm), ref["inv_perm"])
    R, E = cfg.R, cfg.E
    s = i64(layer.ep_splits)
    assert np.array_equal(s[:R * E].reshape(R, E), ref["ep_counts"])
    assert np.array_equal(s[R * E:].reshape(R, R), ref["send_splits"])
    assert np.array_equal(layer.host_splits.numpy().astype(np.int64), s)
    for k in ("send_index", "a2a_index", "regroup_index"):
        assert np.array_equal(i64(getattr(layer, k)), ref[k]), k
    assert np.array_equal(f64(layer.xp), ref["xp"])
    assert_bf16_close(f64(layer.h), ref["h_pre"], name="h")
    assert_bf16_close(f64(layer.gu), ref["gu_pre"], name="gu")
    assert_out_close(f64(layer.y), ref["y_pre"], name="y")
    assert_out_close(f64(out), ref["out_pre"], name="out")
    rb = O.layer_backward(np_inp, ref, np_inp["dout"], cfg.K, cfg.renorm, pre=True)
    assert_out_close(f64(dx), rb["dx_pre"], name="dx")
    assert_out_close(f64(layer.dxp), rb["dxp_pre"], name="dxp")
    assert_rms_close(f64(layer.dlogits), rb["dlogits"], name="dlogits")
    assert_rms_close(f64(layer.dw_gate), rb["dw_gate"], name="dw_gate")
    assert_rms_close(f64(layer.dw_up), rb["dw_up"], name="dw_up")
    assert_rms_close(f64(layer.dw_down), rb["dw_down"], name="dw_down")
    if cfg.shared_I:
        assert_rms_close(f64(layer.dws_gate[0]), rb["dws_gate"], name="dws_gate")
        assert_rms_close(f64(layer.dws_down[0]), rb["dws_down"], name="dws_down")


def test_exactly_one_device_to_host_copy_per_forward():
    cfg = W.small_config("d2h", T=512, d=128, E=16, K=2, I=128, R=4)
    inp = W.make_inputs(cfg, with_backward=False)
    layer = L.layer_from_config(cfg, inp, dev())
    logits, x = inp["logits"].to(dev()), inp["x"].to(dev())
    layer.forward(logits, x)          # warm-up (library load, attribute setup)
    torch.cuda.synchronize()
    from torch.profiler import ProfilerActivity, profile
    from torch.profiler import record_function
    with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]) as prof:
        with record_function("moe_layer_forward"):
            layer.forward(logits, x)
            torch.cuda.synchronize()
    names = [e.name for e in prof.events()]
    d2h = [n for n in names if "Memcpy" in n and ("DtoH" in n or "Device -> " in n)]
    assert len(d2h) == 1, prof.key_averages().table(row_limit=40)
    assert sum(n.startswith("cudaMemcpy") for n in names) == 1, names
