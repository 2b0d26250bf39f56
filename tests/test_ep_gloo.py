"""Both expert-parallel designs over real process groups: 2 and 4 gloo ranks
on the CPU, one process per rank, with ProcessGroupExchange running the count
exchange, the uneven payload all-to-alls (zero-row splits included: one case
leaves a rank with no token to receive), the all-gathers and the
reduce-scatters. Each rank's steps are the CPU stand-ins of the library calls
(the oracle's arithmetic), so what this checks is the host-side choreography
of the exchanges: the gathered per-rank outputs and gradients must equal the
oracle's single-process layer on the whole group's inputs."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


CASES = {
    "r2": dict(T=64, d=32, E=8, K=2, I=32, R=2),
    "r2_idle": dict(T=64, d=32, E=8, K=2, I=32, R=2),
    "r4_shared": dict(T=64, d=32, E=8, K=3, I=32, R=4, shared_I=64),
    "r4_norenorm": dict(T=48, d=32, E=8, K=2, I=32, R=4, renorm=0),
}


def _cfg(name):
    from grouped_gemm_moe_gb300 import workloads as W
    return W.small_config(name, **CASES[name])


def _inputs(name):
    from grouped_gemm_moe_gb300 import workloads as W
    inp = W.make_inputs(_cfg(name), with_backward=True)
    if name == "r2_idle":
        inp["logits"][:, 4:] -= 100.0        # rank 1's experts are never selected
    return inp


def _worker(rank, world, port, name, design, q):
    sys.path[:0] = [ROOT, TESTS]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from grouped_gemm_moe_gb300 import ep as EP
        from _ep_cpu_kernels import CpuKernels
        cfg = _cfg(name)
        inp = _inputs(name)
        Tl = cfg.T // world
        sl = slice(rank * Tl, (rank + 1) * Tl)
        keys = ["w_gate", "w_up", "w_down"] + (["ws_gate", "ws_up", "ws_down"] if cfg.shared_I else [])
        w = EP.local_weights({k: inp[k] for k in keys}, rank, world)
        ex = EP.ProcessGroupExchange()
        lg, x, do = (inp[k][sl].contiguous() for k in ("logits", "x", "dout"))
        Cls = EP.A2ARank if design == "a2a" else EP.AGRSRank
        rk = Cls(rank, world, Tl, cfg.d, cfg.E, cfg.K, cfg.I, w, cfg.renorm, "cpu",
                 kernels=CpuKernels())
        if design == "a2a":
            (out,) = EP.a2a_forward([rk], ex, [lg], [x])
            (dx,) = EP.a2a_backward([rk], ex, [do])
            extra = {"n_recv": rk.n_recv, "send": rk.send_splits, "recv": rk.recv_splits}
        else:
            (out,) = EP.agrs_forward([rk], ex, [lg], [x])
            (dx,) = EP.agrs_backward([rk], ex, [do], [lg])
            extra = {"n_recv": int(rk.local_offsets[-1])}
        # numpy copies: pickled by value, so nothing depends on this process after it exits
        npy = lambda t: t.detach().to(torch.float64).numpy().copy()  # noqa: E731
        res = {k: npy(getattr(rk, k)) for k in ("dlogits", "dw_gate", "dw_up", "dw_down")}
        if cfg.shared_I:
            res["dws_gate"] = npy(rk.dws_gate)
        q.put((rank, npy(out), npy(dx), res, extra, None))
    except Exception as e:  # pragma: no cover - reported by the parent
        import traceback
        q.put((rank, None, None, None, None, traceback.format_exc()))
    finally:
        dist.destroy_process_group()


def _run(name, design):
    cfg = _cfg(name)
    world = cfg.R
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, name, design, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=300) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
    for r in got:
        assert r[5] is None, r[5]
    for p in procs:
        assert p.exitcode == 0
    return cfg, got


@pytest.mark.parametrize("design", ["a2a", "agrs"])
@pytest.mark.parametrize("name", list(CASES))
def test_ep_over_gloo_ranks_matches_oracle(name, design):
    from grouped_gemm_moe_gb300 import workloads as W
    from oracle import moe_oracle as O
    from _parity import assert_out_close, assert_rms_close
    cfg, got = _run(name, design)
    inp = _inputs(name)
    np_inp = {k: W.to_f64(v) for k, v in inp.items()}
    ref = O.layer_forward(np_inp, cfg.K, cfg.R, cfg.renorm, pre=True)
    rb = O.layer_backward(np_inp, ref, np_inp["dout"], cfg.K, cfg.renorm, pre=True)
    cat = lambda i: np.concatenate([g[i] for g in got])  # noqa: E731
    assert_out_close(cat(1), ref["out_pre"], tol=1e-3, name="out")
    assert_out_close(cat(2), rb["dx_pre"], tol=1e-3, name="dx")
    res = lambda k: np.concatenate([g[3][k] for g in got])  # noqa: E731
    assert_rms_close(res("dlogits"), rb["dlogits"], 1e-5, name="dlogits")
    for k in ("dw_gate", "dw_up", "dw_down"):
        assert_rms_close(res(k), rb[k], 1e-5, name=k)
    if cfg.shared_I:
        dws = sum(g[3]["dws_gate"][0] for g in got)
        assert_rms_close(dws, rb["dws_gate"], 1e-5, name="dws_gate")
    El = cfg.E // cfg.R
    off = ref["offsets"]
    for r, g in enumerate(got):
        assert g[4]["n_recv"] == off[(r + 1) * El] - off[r * El]
        if design == "a2a":
            S = ref["send_splits"]
            assert g[4]["send"] == S[r].tolist() and g[4]["recv"] == S[:, r].tolist()
    if name == "r2_idle":
        assert got[1][4]["n_recv"] == 0
        assert (got[1][3]["dw_gate"] == 0).all()
