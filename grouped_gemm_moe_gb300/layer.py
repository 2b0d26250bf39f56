"""One MoE layer's forward and backward on one GPU, as a fixed sequence of
library calls on the current CUDA stream with every buffer preallocated.

Forward:  moe_route_permute_ep (router top-k, the permutation and
          the simulated expert-parallel layout from one pass, with the one
          device-to-host copy of the splits) -> moe_dispatch_scatter ->
          moe_grouped_ffn (routed experts; shared experts as E=1 on x) ->
          moe_combine.
Backward: moe_combine_backward -> moe_grouped_ffn_backward_data (routed; shared)
          -> moe_dispatch_backward -> moe_grouped_ffn_backward_weights (routed;
          shared) -> moe_route_topk_backward.

With aux_loss_coef > 0 the forward also runs moe_load_balance (per-expert load
fractions, mean router probabilities, the load-balance loss and load metrics,
in lb_frac / lb_pmean / lb_stats) and the backward adds aux_loss_coef times
the loss's gradient into dlogits with moe_load_balance_backward.

This module only allocates tensors and orders the calls; each step is a
kernel of libmoe_gb300.so.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import torch

from . import binding as B


class MoELayer:
    def __init__(self, T: int, d: int, E: int, K: int, I: int, R: int,
                 weights: Dict[str, torch.Tensor], renorm: int = 1,
                 device: Optional[torch.device] = None, aux_loss_coef: float = 0.0):
        self.T, self.d, self.E, self.K, self.I, self.R = T, d, E, K, I, R
        self.renorm = renorm
        dev = torch.device(device) if device is not None else weights["w_gate"].device
        self.device = dev
        self.w = weights
        self.shared = "ws_gate" in weights
        TK = T * K
        bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        # forward buffers
        self.topk_idx, self.topk_w = e(T, K, dt=i32), e(T, K, dt=f32)
        self.counts, self.offsets = e(E, dt=i32), e(E + 1, dt=i32)
        self.perm, self.inv_perm = e(TK, dt=i32), e(TK, dt=i32)
        n_split = R * E + R * R
        self.ep_splits = e(n_split, dt=i32)
        self.send_index, self.a2a_index, self.regroup_index = (e(TK, dt=i32) for _ in range(3))
        self.host_splits = torch.empty(n_split, dtype=i32, pin_memory=True)
        self.xp = e(TK, d, dt=bf)
        self.y, self.h, self.gu = e(TK, d, dt=bf), e(TK, I, dt=bf), e(TK, 2 * I, dt=bf)
        self.out = e(T, d, dt=bf)
        self.ws_ep = B.new_workspace(B.workspace_size(B.MOE_OP_ROUTE_PERMUTE_EP, T, E, K, R), dev)
        self.ws_ffn = B.new_workspace(B.workspace_size(B.MOE_OP_GROUPED_FFN, T, E, K, 1, d, I), dev)
        # backward buffers
        self.dy, self.dtopk_w = e(TK, d, dt=bf), e(T, K, dt=f32)
        self.dxp = e(TK, d, dt=bf)
        self.dw_gate, self.dw_up = e(E, d, I, dt=f32), e(E, d, I, dt=f32)
        self.dw_down = e(E, I, d, dt=f32)
        self.dx, self.dlogits = e(T, d, dt=bf), e(T, E, dt=f32)
        self.ws_bwd = B.new_workspace(
            B.workspace_size(B.MOE_OP_GROUPED_FFN_BACKWARD, T, E, K, 1, d, I), dev)
        if self.shared:
            Is = weights["ws_gate"].shape[1]
            self.Is = Is
            self.ws_g = weights["ws_gate"].unsqueeze(0)
            self.ws_u = weights["ws_up"].unsqueeze(0)
            self.ws_d = weights["ws_down"].unsqueeze(0)
            self.s_offsets = torch.tensor([0, T], dtype=i32, device=dev)
            self.ys, self.hs, self.gus = e(T, d, dt=bf), e(T, Is, dt=bf), e(T, 2 * Is, dt=bf)
            self.dxs = e(T, d, dt=bf)
            self.dws_gate, self.dws_up = e(1, d, Is, dt=f32), e(1, d, Is, dt=f32)
            self.dws_down = e(1, Is, d, dt=f32)
            self.ws_sfwd = B.new_workspace(B.workspace_size(B.MOE_OP_GROUPED_FFN, T, 1, 1, 1, d, Is), dev)
            self.ws_sbwd = B.new_workspace(
                B.workspace_size(B.MOE_OP_GROUPED_FFN_BACKWARD, T, 1, 1, 1, d, Is), dev)
        self.aux_loss_coef = float(aux_loss_coef)
        if self.aux_loss_coef > 0:
            self.lb_frac, self.lb_pmean, self.lb_stats = e(E, dt=f32), e(E, dt=f32), e(4, dt=f32)
            self.ws_lb = B.new_workspace(B.workspace_size(B.MOE_OP_LOAD_BALANCE, T, E, K), dev)
        self.logits = None
        self.x = None
        self.timeline: Optional[List] = None   # when a list, (name, start_event, end_event) per call
        self._mark_splits = False
        self.splits_issued = None

    # -------------------------------------------------------------- timing hooks
    def _mark(self, name):
        if self.timeline is None:
            return None
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(torch.cuda.current_stream(self.device))
        return (name, ev)

    def _close(self, tok):
        if tok is None:
            return
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(torch.cuda.current_stream(self.device))
        self.timeline.append((tok[0], tok[1], ev))

    def _run(self, name, fn, *a, **k):
        tok = self._mark(name)
        r = fn(*a, **k)
        self._close(tok)
        return r

    # -------------------------------------------------------------- passes
    def forward(self, logits: torch.Tensor, x: torch.Tensor, copy_splits: bool = True):
        self.logits, self.x = logits, x
        w = self.w
        K, E, R = self.K, self.E, self.R
        self._run("route_permute_ep", B.moe_route_permute_ep, logits, K, R, self.renorm,
                  host_splits=self.host_splits if copy_splits else False, ws=self.ws_ep,
                  out=(self.topk_idx, self.topk_w, self.counts, self.offsets, self.perm,
                       self.inv_perm, self.ep_splits, self.send_index, self.a2a_index,
                       self.regroup_index))
        if self.aux_loss_coef > 0:
            self._run("load_balance", B.moe_load_balance, logits, self.counts, K, ws=self.ws_lb,
                      out=(self.lb_frac, self.lb_pmean, self.lb_stats))
        if self._mark_splits:   # the splits' device-to-host copy has been issued
            self.splits_issued = torch.cuda.Event()
            self.splits_issued.record(torch.cuda.current_stream(self.device))
        self._run("dispatch", B.moe_dispatch_scatter, x, self.inv_perm, K, out=self.xp)
        self._run("grouped_ffn", B.moe_grouped_ffn, self.xp, self.offsets, w["w_gate"], w["w_up"],
                  w["w_down"], ws=self.ws_ffn, out=(self.y, self.h, self.gu))
        shared_y = None
        if self.shared:
            self._run("shared_ffn", B.moe_grouped_ffn, x, self.s_offsets, self.ws_g, self.ws_u,
                      self.ws_d, ws=self.ws_sfwd, out=(self.ys, self.hs, self.gus))
            shared_y = self.ys
        self._run("combine", B.moe_combine, self.y, self.topk_w, self.inv_perm, shared_y,
                  out=self.out)
        return self.out

    def backward(self, dout: torch.Tensor):
        w = self.w
        self._run("combine_backward", B.moe_combine_backward, dout, self.y, self.topk_w,
                  self.inv_perm, out=(self.dy, self.dtopk_w))
        # data parts first, then the gather of dx while the GEMMs' dX rows are still
        # in L2, then the weight gradients
        self._run("grouped_ffn_backward_data", B.moe_grouped_ffn_backward_data, self.dy, self.xp,
                  self.gu, self.h, self.offsets, w["w_gate"], w["w_up"], w["w_down"],
                  ws=self.ws_bwd, out=self.dxp)
        dxs = None
        if self.shared:
            self._run("shared_ffn_backward_data", B.moe_grouped_ffn_backward_data, dout, self.x,
                      self.gus, self.hs, self.s_offsets, self.ws_g, self.ws_u, self.ws_d,
                      ws=self.ws_sbwd, out=self.dxs)
            dxs = self.dxs
        self._run("dispatch_backward", B.moe_dispatch_backward, self.dxp, self.inv_perm, self.T,
                  self.K, dxs, out=self.dx)
        self._run("grouped_ffn_backward_weights", B.moe_grouped_ffn_backward_weights, self.dy,
                  self.xp, self.h, self.offsets, self.E, self.I, ws=self.ws_bwd,
                  out=(self.dw_gate, self.dw_up, self.dw_down))
        if self.shared:
            self._run("shared_ffn_backward_weights", B.moe_grouped_ffn_backward_weights, dout,
                      self.x, self.hs, self.s_offsets, 1, self.Is, ws=self.ws_sbwd,
                      out=(self.dws_gate, self.dws_up, self.dws_down))
        self._run("route_topk_backward", B.moe_route_topk_backward,
                  None if self.renorm else self.logits, self.topk_idx, self.topk_w, self.dtopk_w,
                  self.E, self.renorm, out=self.dlogits)
        if self.aux_loss_coef > 0:
            self._run("load_balance_backward", B.moe_load_balance_backward, self.logits,
                      self.lb_frac, self.aux_loss_coef, dlogits=self.dlogits, accumulate=True)
        return self.dx

    def step_from_host(self, logits_h: torch.Tensor, x_h: torch.Tensor, dout_h: torch.Tensor,
                       out_h: torch.Tensor, dx_h: torch.Tensor):
        """One forward + backward whose inputs start in (pinned) host memory and
        whose outputs end there. logits and x are copied in on the current
        stream; dout is copied in on a side stream while the forward runs, and
        the output is copied out on the side stream while the backward runs.
        The current stream joins the side stream before returning, so work
        enqueued after this call sees every copy finished. Returns the bytes
        copied each way."""
        dev = self.device
        if not hasattr(self, "_in_logits"):
            self._in_logits = torch.empty(self.T, self.E, dtype=torch.float32, device=dev)
            self._in_x = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=dev)
            self._in_dout = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=dev)
            self._side = torch.cuda.Stream(device=dev)
        cur = torch.cuda.current_stream(dev)
        side = self._side
        side.wait_stream(cur)                 # earlier readers of _in_dout / out are done
        self._in_logits.copy_(logits_h, non_blocking=True)
        self._in_x.copy_(x_h, non_blocking=True)
        with torch.cuda.stream(side):
            self._in_dout.copy_(dout_h, non_blocking=True)
            dout_ready = torch.cuda.Event()
            dout_ready.record(side)
        out = self.forward(self._in_logits, self._in_x)
        fwd_done = torch.cuda.Event()
        fwd_done.record(cur)
        with torch.cuda.stream(side):
            side.wait_event(fwd_done)
            out_h.copy_(out, non_blocking=True)
        cur.wait_event(dout_ready)
        dx = self.backward(self._in_dout)
        dx_h.copy_(dx, non_blocking=True)
        cur.wait_stream(side)
        h2d = logits_h.numel() * 4 + x_h.numel() * 2 + dout_h.numel() * 2
        d2h = out_h.numel() * 2 + dx_h.numel() * 2 + self.host_splits.numel() * 4
        return h2d, d2h

    def run_from_host(self, steps):
        """A sequence of forward + backward steps whose inputs start in pinned
        host memory and whose outputs end there. ``steps`` is a list of
        ``(logits_h, x_h, dout_h, out_h, dx_h)``.

        Inputs go to the device through two alternating input slots on an
        upload stream, so step i+1's copy runs while step i computes; out and
        dx go back on a download stream while the next pass runs. The large
        copies are issued only after the step's own small copy of the EP
        splits (on the compute stream), so that copy never queues behind a
        33 MB transfer. Every step still moves its own inputs in and its
        outputs out. The current stream joins both copy streams before
        returning. Returns the bytes copied each way per step (of the last
        step)."""
        dev = self.device
        if not hasattr(self, "_slots"):
            bf = torch.bfloat16
            self._slots = [(torch.empty(self.T, self.E, dtype=torch.float32, device=dev),
                            torch.empty(self.T, self.d, dtype=bf, device=dev),
                            torch.empty(self.T, self.d, dtype=bf, device=dev)) for _ in range(2)]
            self._up = torch.cuda.Stream(device=dev)
            self._down = torch.cuda.Stream(device=dev)
        cur = torch.cuda.current_stream(dev)
        up, down = self._up, self._down
        up.wait_stream(cur)      # earlier readers of the slots and of out / dx are done
        down.wait_stream(cur)
        n = len(steps)
        in_ready = [None] * n

        def after(stream):
            ev = torch.cuda.Event()
            ev.record(stream)
            return ev

        def upload(i, gate=None):
            with torch.cuda.stream(up):
                if gate is not None:
                    up.wait_event(gate)
                for dst, src in zip(self._slots[i % 2], steps[i][:3]):
                    dst.copy_(src, non_blocking=True)
                in_ready[i] = after(up)

        if n:
            upload(0)
        out_copied = dx_copied = None
        pending_dx = None        # the previous step's dx_h, downloaded once this step's splits left
        self._mark_splits = True
        try:
            for i in range(n):
                logits, x, dout = self._slots[i % 2]
                out_h, dx_h = steps[i][3], steps[i][4]
                cur.wait_event(in_ready[i])
                if out_copied is not None:
                    cur.wait_event(out_copied)      # the previous step's out has left the device
                out = self.forward(logits, x)
                splits = self.splits_issued      # after the previous backward, in stream order
                fwd_done = after(cur)
                with torch.cuda.stream(down):
                    if pending_dx is not None:
                        down.wait_event(splits)
                        pending_dx.copy_(self.dx, non_blocking=True)
                        dx_copied = after(down)
                    down.wait_event(fwd_done)
                    out_h.copy_(out, non_blocking=True)
                    out_copied = after(down)
                if i + 1 < n:
                    upload(i + 1, gate=splits)   # slot (i+1) % 2 was last read by step i-1
                if dx_copied is not None:
                    cur.wait_event(dx_copied)       # the previous dx has left before it is rewritten
                self.backward(dout)
                pending_dx = dx_h
            if pending_dx is not None:
                with torch.cuda.stream(down):
                    down.wait_stream(cur)
                    pending_dx.copy_(self.dx, non_blocking=True)
        finally:
            self._mark_splits = False
        cur.wait_stream(down)
        cur.wait_stream(up)
        if not n:
            return 0, 0
        lh, xh, dh, oh, dxh = steps[-1]
        h2d = lh.numel() * 4 + xh.numel() * 2 + dh.numel() * 2
        d2h = oh.numel() * 2 + dxh.numel() * 2 + self.host_splits.numel() * 4
        return h2d, d2h

    def device_status(self) -> int:
        """First nonzero device status among the GEMM workspaces (synchronises)."""
        wss = [self.ws_ffn, self.ws_bwd] + ([self.ws_sfwd, self.ws_sbwd] if self.shared else [])
        for ws in wss:
            s = B.moe_read_device_status(ws)
            if s:
                return s
        return 0


def layer_from_config(cfg, inputs: Dict[str, torch.Tensor], device,
                      aux_loss_coef: float = 0.0) -> MoELayer:
    """Copies a workload's weights to ``device`` and builds the layer."""
    keys = ["w_gate", "w_up", "w_down"] + (["ws_gate", "ws_up", "ws_down"] if cfg.shared_I else [])
    weights = {k: inputs[k].to(device).contiguous() for k in keys}
    return MoELayer(cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.R, weights, cfg.renorm, device,
                    aux_loss_coef)
