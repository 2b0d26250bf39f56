"""The debug-checks build (-DMOE_DEBUG_CHECKS, libmoe_gb300_debug.so) in a
child process: on valid inputs it records no failed check and gives exactly
the release library's results for a whole layer forward + backward; given an
inv_perm entry past the packed rows, the combine's check records
MOE_ERR_DEVICE_CHECK and reads row 0 instead (the other tokens unchanged)."""
import multiprocessing as mp
import os
import sys

import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import layer as L
from grouped_gemm_moe_gb300 import workloads as W

from _parity import dev, ensure_built

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CFG = dict(T=512, d=256, E=16, K=4, I=256, R=4)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _layer_outputs():
    cfg = W.small_config("dbg", **CFG)
    inp = W.make_inputs(cfg, with_backward=True)
    layer = L.layer_from_config(cfg, inp, dev())
    out = layer.forward(inp["logits"].to(dev()), inp["x"].to(dev())).clone()
    dx = layer.backward(inp["dout"].to(dev())).clone()
    torch.cuda.synchronize()
    res = {"out": out, "dx": dx, "dlogits": layer.dlogits, "dw_gate": layer.dw_gate,
           "perm": layer.perm, "regroup_index": layer.regroup_index}
    return {k: v.cpu().to(torch.float64).numpy() for k, v in res.items()}, layer.device_status()


def _child(q):
    sys.path.insert(0, ROOT)
    try:
        from grouped_gemm_moe_gb300 import binding as B
        from grouped_gemm_moe_gb300 import build as build_mod
        B.load(build_mod.build(debug=True))
        res, status = _layer_outputs()
        clean = B.moe_debug_check_status()
        # an out-of-range position in the combine's inv_perm
        T, K, d = 64, 2, 64
        g = torch.Generator().manual_seed(3)
        y = torch.randn(T * K, d, generator=g).to(torch.bfloat16).to(dev())
        w = torch.rand(T, K, generator=g).to(dev())
        inv = torch.arange(T * K, dtype=torch.int32)
        good = B.moe_combine(y, w, inv.to(dev()))
        bad_inv = inv.clone()
        bad_inv[5 * K + 1] = T * K + 1000
        bad = B.moe_combine(y, w, bad_inv.to(dev()))
        torch.cuda.synchronize()
        flagged = B.moe_debug_check_status()
        after = B.moe_debug_check_status()
        f = lambda t: t.cpu().to(torch.float64).numpy()  # noqa: E731
        q.put((res, status, clean, flagged, after, f(good), f(bad), None))
    except Exception:  # pragma: no cover - reported by the parent
        import traceback
        q.put((None,) * 7 + (traceback.format_exc(),))


def test_debug_build_matches_release_and_flags_a_bad_index():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_child, args=(q,))
    p.start()
    res, status, clean, flagged, after, good, bad, err = q.get(timeout=600)
    p.join(timeout=60)
    assert err is None, err
    assert p.exitcode == 0
    assert status == 0 and clean == 0
    rel, _ = _layer_outputs()
    for k, v in rel.items():
        assert np.array_equal(res[k], v), k
    assert flagged == 7 and after == 0            # MOE_ERR_DEVICE_CHECK, then cleared
    T, K = 64, 2
    keep = np.ones(T, bool)
    keep[5] = False
    assert np.array_equal(good[keep], bad[keep])
    assert not np.array_equal(good[5], bad[5])


def test_release_build_reports_unsupported():
    from grouped_gemm_moe_gb300 import binding as B
    with pytest.raises(B.MoEError) as ei:
        B.moe_debug_check_status()
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
