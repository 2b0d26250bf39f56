"""Expert parallelism over real ranks: one MoE layer whose routed experts are
split over R ranks, each rank holding T_local tokens and E/R experts.

Two designs from the pages, both built from the library's kernels:

* ``A2ARank`` -- all-to-all EP ("Three axes of Parallelism" (nanoTitan blog),
  "Expert Parallel (EP)" -> "Dispatch, expert computation and combine";
  modalities PR "expert parallelism for the Nemotron-3 Nano MoE layers",
  "Design" items 1-2). Each rank routes its own tokens and packs them
  expert-major (that packed buffer is the send buffer); the per-expert counts
  are exchanged; the receive-side layout kernel writes both split lists, the
  local expert offsets and the regroup index, and one device-to-host copy
  brings the split lists to the host for the payload all-to-all. The received
  rows are regrouped by local expert, run through the grouped SwiGLU GEMM,
  put back in receive order and sent back; the combine then reads them in
  the rank's own packed order. The backward runs the same exchanges with the
  gradients.
* ``AGRSRank`` -- all-gather / reduce-scatter EP (SpecForge PR "expert
  parallelism for MoE drafters on the FSDP2 backend", "What this adds", the
  MoELayer.forward under EP bullet). Every rank all-gathers the group's router
  logits and tokens, runs the replicated router on all of them, gathers only
  the rows of its own experts, runs them, and combines them into fp32
  partial outputs of every token; a reduce-scatter sums the partials onto the
  tokens' owners, which add the shared expert and round to bf16. The backward
  all-gathers the upstream gradient and reduce-scatters the fp32 input
  gradient and the router-weight gradient.

The collectives are an ``Exchange``: ``ProcessGroupExchange`` runs them with
torch.distributed (one rank per process: NCCL between GPUs, gloo on CPU);
``LoopbackExchange`` drives all R ranks of a group from one process on one
device and moves the rows with device copies, which lets one GPU run the
whole multi-rank data path. ``a2a_forward`` / ``a2a_backward`` and
``agrs_forward`` / ``agrs_backward`` run a list of ranks (one, or all R)
step by step with the exchanges between the steps.

Each rank calls its kernels through ``kernels`` (default: the CUDA library
binding, which raises on non-CUDA tensors; there is no CPU path in this
package). Sender partition: rank r holds tokens [r*T_local, (r+1)*T_local) of
the group and experts [r*E/R, (r+1)*E/R).
"""
from __future__ import annotations

import abc
from typing import Dict, List, Sequence

import torch

from . import binding as B


class CudaKernels:
    """The per-rank steps: the library's entry points (argument marshalling only)."""

    route_topk = staticmethod(B.moe_route_topk)
    route_topk_backward = staticmethod(B.moe_route_topk_backward)
    build_permutation = staticmethod(B.moe_build_permutation)
    dispatch = staticmethod(B.moe_dispatch)
    dispatch_scatter = staticmethod(B.moe_dispatch_scatter)
    ep_recv_layout = staticmethod(B.moe_ep_recv_layout)
    grouped_ffn = staticmethod(B.moe_grouped_ffn)
    grouped_ffn_backward_data = staticmethod(B.moe_grouped_ffn_backward_data)
    grouped_ffn_backward_weights = staticmethod(B.moe_grouped_ffn_backward_weights)
    combine = staticmethod(B.moe_combine)
    combine_backward = staticmethod(B.moe_combine_backward)
    dispatch_backward = staticmethod(B.moe_dispatch_backward)
    dispatch_slice = staticmethod(B.moe_dispatch_slice)
    combine_slice = staticmethod(B.moe_combine_slice)
    combine_backward_slice = staticmethod(B.moe_combine_backward_slice)
    dispatch_backward_slice = staticmethod(B.moe_dispatch_backward_slice)
    reduce_finish = staticmethod(B.moe_reduce_finish)

    @staticmethod
    def workspace(op, T, E, K, R, d, I, device, zero: bool = False):
        ws = B.new_workspace(B.workspace_size(op, T, E, K, R, d, I), device)
        if zero:
            ws.zero_()
        return ws


# --------------------------------------------------------------------- exchanges
class Exchange(abc.ABC):
    """Collectives of one EP group over the ranks this process drives: each
    argument is a list with one tensor per driven rank, in ``ranks`` order."""

    R: int
    ranks: List[int]

    @abc.abstractmethod
    def all_to_all_equal(self, sends: Sequence[torch.Tensor]) -> List[torch.Tensor]:
        """Each send holds R equal chunks; chunk q goes to rank q. Returns, per
        driven rank, the R chunks it received, in source order."""

    @abc.abstractmethod
    def all_to_all(self, recvs, sends, recv_splits, send_splits) -> None:
        """Row all-to-all: send rows [sum(send_splits[:q]), ...) go to rank q and
        land in its recv at the source's block (recv_splits per source)."""

    @abc.abstractmethod
    def all_gather(self, outs, ins) -> None:
        """outs[i] = the concatenation of every rank's in, in rank order."""

    @abc.abstractmethod
    def reduce_scatter(self, outs, ins) -> None:
        """outs[i] = block ``ranks[i]`` of the element-wise sum of every rank's in."""


class ProcessGroupExchange(Exchange):
    """One rank per process over a torch.distributed process group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.R = dist.get_world_size(group)
        self.ranks = [dist.get_rank(group)]

    def all_to_all_equal(self, sends):
        (send,) = sends
        recv = torch.empty_like(send)
        self.dist.all_to_all_single(recv, send, group=self.group)
        return [recv]

    def all_to_all(self, recvs, sends, recv_splits, send_splits):
        self.dist.all_to_all_single(recvs[0], sends[0], output_split_sizes=list(recv_splits[0]),
                                    input_split_sizes=list(send_splits[0]), group=self.group)

    def all_gather(self, outs, ins):
        self.dist.all_gather_into_tensor(outs[0], ins[0], group=self.group)

    def reduce_scatter(self, outs, ins):
        self.dist.reduce_scatter_tensor(outs[0], ins[0], op=self.dist.ReduceOp.SUM, group=self.group)


class LoopbackExchange(Exchange):
    """All R ranks of the group in this process: the collectives are device
    copies between the ranks' buffers (and a sum for the reduce-scatter), in
    stream order on the current stream."""

    def __init__(self, R: int):
        self.R = R
        self.ranks = list(range(R))

    def all_to_all_equal(self, sends):
        R = self.R
        c = sends[0].numel() // R
        m = torch.stack([s.view(R, c) for s in sends])          # [source, destination, c]
        return [m[:, q].contiguous().view(-1) for q in range(R)]

    def all_to_all(self, recvs, sends, recv_splits, send_splits):
        R = self.R
        for s in range(R):
            so = 0
            for q in range(R):
                n = int(send_splits[s][q])
                if n:
                    ro = sum(int(v) for v in recv_splits[q][:s])
                    recvs[q][ro:ro + n].copy_(sends[s][so:so + n])
                so += n

    def all_gather(self, outs, ins):
        whole = torch.cat(list(ins))
        for o in outs:
            o.copy_(whole)

    def reduce_scatter(self, outs, ins):
        total = torch.stack(list(ins)).sum(0)
        n = outs[0].shape[0]
        for r, o in zip(self.ranks, outs):
            o.copy_(total[r * n:(r + 1) * n])


# --------------------------------------------------------------------- all-to-all EP
class A2ARank:
    """One rank of all-to-all EP: T_local tokens, experts [rank*El, (rank+1)*El)
    with their weights ``w_gate``, ``w_up`` [El,d,I] and ``w_down`` [El,I,d]
    (optional shared-expert weights ``ws_gate``, ``ws_up`` [d,Is], ``ws_down``
    [Is,d], applied to the rank's own tokens)."""

    def __init__(self, rank: int, R: int, T_local: int, d: int, E: int, K: int, I: int,
                 weights: Dict[str, torch.Tensor], renorm: int = 1, device=None, kernels=None):
        if E % R:
            raise ValueError("R must divide E")
        self.k = kernels or CudaKernels()
        self.rank, self.R, self.T, self.d, self.E, self.K, self.I = rank, R, T_local, d, E, K, I
        self.El = E // R
        self.renorm = renorm
        dev = torch.device(device) if device is not None else weights["w_gate"].device
        self.device = dev
        self.w = weights
        self.shared = "ws_gate" in weights
        TK = T_local * K
        # every source sends at most T_local * min(K, El) rows to this rank
        self.cap = R * T_local * min(K, self.El)
        bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.topk_idx, self.topk_w = e(T_local, K, dt=i32), e(T_local, K, dt=f32)
        self.counts, self.offsets = e(E, dt=i32), e(E + 1, dt=i32)
        self.perm, self.inv_perm = e(TK, dt=i32), e(TK, dt=i32)
        self.send_buf = e(TK, d, dt=bf)
        self.splits, self.local_offsets = e(2 * R, dt=i32), e(self.El + 1, dt=i32)
        self.regroup = e(max(self.cap, 1), dt=i32)
        pin = dev.type == "cuda"
        self.host_splits = torch.empty(2 * R, dtype=i32, pin_memory=pin)
        cap = max(self.cap, 1)
        self.recv_buf, self.xe = e(cap, d, dt=bf), e(cap, d, dt=bf)
        self.y, self.h, self.gu = e(cap, d, dt=bf), e(cap, I, dt=bf), e(cap, 2 * I, dt=bf)
        self.yr, self.ret_buf = e(cap, d, dt=bf), e(TK, d, dt=bf)
        self.out = e(T_local, d, dt=bf)
        self.ws_perm = self.k.workspace(B.MOE_OP_BUILD_PERMUTATION, T_local, E, K, 1, 0, 0, dev)
        self.ws_recv = self.k.workspace(B.MOE_OP_EP_RECV_LAYOUT, 1, E, 1, R, 0, 0, dev)
        self.ws_ffn = self.k.workspace(B.MOE_OP_GROUPED_FFN, cap, self.El, 1, 1, d, I, dev)
        self.ws_bwd = self.k.workspace(B.MOE_OP_GROUPED_FFN_BACKWARD, cap, self.El, 1, 1, d, I, dev)
        # backward
        self.dys, self.dtopk_w = e(TK, d, dt=bf), e(T_local, K, dt=f32)
        self.dyr, self.dye, self.dxe, self.dxr = (e(cap, d, dt=bf) for _ in range(4))
        self.dxs = e(TK, d, dt=bf)
        self.dx, self.dlogits = e(T_local, d, dt=bf), e(T_local, E, dt=f32)
        El = self.El
        self.dw_gate, self.dw_up = e(El, d, I, dt=f32), e(El, d, I, dt=f32)
        self.dw_down = e(El, I, d, dt=f32)
        if self.shared:
            Is = weights["ws_gate"].shape[1]
            self.Is = Is
            self.ws_g, self.ws_u, self.ws_d = (weights[k].unsqueeze(0)
                                               for k in ("ws_gate", "ws_up", "ws_down"))
            self.s_offsets = torch.tensor([0, T_local], dtype=i32, device=dev)
            self.ys, self.hs, self.gus = e(T_local, d, dt=bf), e(T_local, Is, dt=bf), e(T_local, 2 * Is, dt=bf)
            self.dx_shared = e(T_local, d, dt=bf)
            self.dws_gate, self.dws_up = e(1, d, Is, dt=f32), e(1, d, Is, dt=f32)
            self.dws_down = e(1, Is, d, dt=f32)
            self.ws_sfwd = self.k.workspace(B.MOE_OP_GROUPED_FFN, T_local, 1, 1, 1, d, Is, dev)
            self.ws_sbwd = self.k.workspace(B.MOE_OP_GROUPED_FFN_BACKWARD, T_local, 1, 1, 1, d, Is,
                                            dev)
        self.n_recv = 0
        self.send_splits: List[int] = []
        self.recv_splits: List[int] = []
        self._splits_ready = None

    # forward steps -------------------------------------------------------
    def route_and_pack(self, logits: torch.Tensor, x: torch.Tensor) -> torch.Tensor:
        """Route this rank's tokens, pack them expert-major into the send buffer;
        returns the per-expert counts for the count exchange."""
        k = self.k
        self.logits, self.x = logits, x
        k.route_topk(logits, self.K, self.renorm, out=(self.topk_idx, self.topk_w))
        k.build_permutation(self.topk_idx, self.E, ws=self.ws_perm,
                            out=(self.counts, self.offsets, self.perm, self.inv_perm))
        k.dispatch_scatter(x, self.inv_perm, self.K, out=self.send_buf)
        return self.counts

    def layout(self, recv_counts: torch.Tensor) -> None:
        """Receive-side layout from the exchanged counts, and the one
        device-to-host copy of both split lists."""
        self.recv_counts = recv_counts
        self.k.ep_recv_layout(self.counts, recv_counts, self.R, self.cap,
                              host_splits=self.host_splits, ws=self.ws_recv,
                              out=(self.splits, self.local_offsets, self.regroup))
        if self.device.type == "cuda":
            self._splits_ready = torch.cuda.Event()
            self._splits_ready.record(torch.cuda.current_stream(self.device))

    def read_splits(self) -> None:
        """Waits for the split copy; the host split lists of the payload exchange."""
        if self._splits_ready is not None:
            self._splits_ready.synchronize()
        h = self.host_splits.tolist()
        self.send_splits, self.recv_splits = h[:self.R], h[self.R:]
        self.n_recv = sum(self.recv_splits)

    def experts(self) -> None:
        """Regroup the received rows by local expert, run the experts, and put the
        outputs back in receive order for the return exchange."""
        k, n = self.k, self.n_recv
        w = self.w
        if n:
            reg = self.regroup[:n]
            k.dispatch(self.recv_buf[:n], reg, 1, out=self.xe[:n])
        k.grouped_ffn(self.xe[:n], self.local_offsets, w["w_gate"], w["w_up"], w["w_down"],
                      ws=self.ws_ffn, out=(self.y[:n], self.h[:n], self.gu[:n]))
        if n:
            k.dispatch_scatter(self.y[:n], self.regroup[:n], 1, out=self.yr[:n])

    def combine(self) -> torch.Tensor:
        k = self.k
        shared_y = None
        if self.shared:
            k.grouped_ffn(self.x, self.s_offsets, self.ws_g, self.ws_u, self.ws_d, ws=self.ws_sfwd,
                          out=(self.ys, self.hs, self.gus))
            shared_y = self.ys
        k.combine(self.ret_buf, self.topk_w, self.inv_perm, shared_y, out=self.out)
        return self.out

    # backward steps ------------------------------------------------------
    def combine_backward(self, dout: torch.Tensor) -> None:
        self.dout = dout
        self.k.combine_backward(dout, self.ret_buf, self.topk_w, self.inv_perm,
                                out=(self.dys, self.dtopk_w))

    def experts_backward(self) -> None:
        """Regroup the received output gradients, the experts' data and weight
        gradients, and the input gradients back in receive order."""
        k, n, w = self.k, self.n_recv, self.w
        if n:
            k.dispatch(self.dyr[:n], self.regroup[:n], 1, out=self.dye[:n])
        k.grouped_ffn_backward_data(self.dye[:n], self.xe[:n], self.gu[:n], self.h[:n],
                                    self.local_offsets, w["w_gate"], w["w_up"], w["w_down"],
                                    ws=self.ws_bwd, out=self.dxe[:n])
        if n:
            k.dispatch_scatter(self.dxe[:n], self.regroup[:n], 1, out=self.dxr[:n])
        k.grouped_ffn_backward_weights(self.dye[:n], self.xe[:n], self.h[:n], self.local_offsets,
                                       self.El, self.I, ws=self.ws_bwd,
                                       out=(self.dw_gate, self.dw_up, self.dw_down))

    def dispatch_backward(self) -> torch.Tensor:
        k = self.k
        dxs = None
        if self.shared:
            k.grouped_ffn_backward_data(self.dout, self.x, self.gus, self.hs, self.s_offsets,
                                        self.ws_g, self.ws_u, self.ws_d, ws=self.ws_sbwd,
                                        out=self.dx_shared)
            k.grouped_ffn_backward_weights(self.dout, self.x, self.hs, self.s_offsets, 1, self.Is,
                                           ws=self.ws_sbwd,
                                           out=(self.dws_gate, self.dws_up, self.dws_down))
            dxs = self.dx_shared
        k.dispatch_backward(self.dxs, self.inv_perm, self.T, self.K, dxs, out=self.dx)
        k.route_topk_backward(None if self.renorm else self.logits, self.topk_idx, self.topk_w,
                              self.dtopk_w, self.E, self.renorm, out=self.dlogits)
        return self.dx


def a2a_forward(ranks: Sequence[A2ARank], ex: Exchange, logits: Sequence[torch.Tensor],
                xs: Sequence[torch.Tensor]) -> List[torch.Tensor]:
    """Forward of all-to-all EP for the ranks this process drives (``ex.ranks``):
    route and pack, count exchange, receive layout (one host copy of the
    splits), payload exchange, experts, return exchange, combine."""
    counts = [rk.route_and_pack(lg, x) for rk, lg, x in zip(ranks, logits, xs)]
    recv_counts = ex.all_to_all_equal(counts)
    for rk, rc in zip(ranks, recv_counts):
        rk.layout(rc)
    for rk in ranks:
        rk.read_splits()
    ex.all_to_all([rk.recv_buf[:rk.n_recv] for rk in ranks], [rk.send_buf for rk in ranks],
                  [rk.recv_splits for rk in ranks], [rk.send_splits for rk in ranks])
    for rk in ranks:
        rk.experts()
    ex.all_to_all([rk.ret_buf for rk in ranks], [rk.yr[:rk.n_recv] for rk in ranks],
                  [rk.send_splits for rk in ranks], [rk.recv_splits for rk in ranks])
    return [rk.combine() for rk in ranks]


def a2a_backward(ranks: Sequence[A2ARank], ex: Exchange,
                 douts: Sequence[torch.Tensor]) -> List[torch.Tensor]:
    """Backward of all-to-all EP: the combine's backward, the output gradients
    out to the experts' owners, the experts' backward, the input gradients
    back, the dispatch's and router's backward."""
    for rk, do in zip(ranks, douts):
        rk.combine_backward(do)
    ex.all_to_all([rk.dyr[:rk.n_recv] for rk in ranks], [rk.dys for rk in ranks],
                  [rk.recv_splits for rk in ranks], [rk.send_splits for rk in ranks])
    for rk in ranks:
        rk.experts_backward()
    ex.all_to_all([rk.dxs for rk in ranks], [rk.dxr[:rk.n_recv] for rk in ranks],
                  [rk.send_splits for rk in ranks], [rk.recv_splits for rk in ranks])
    return [rk.dispatch_backward() for rk in ranks]


# --------------------------------------------------------------------- all-gather / reduce-scatter EP
class AGRSRank:
    """One rank of all-gather / reduce-scatter EP: T_local tokens of a group of
    R * T_local, experts [rank*El, (rank+1)*El) with their weights (as
    A2ARank), optional shared expert on the rank's own tokens."""

    def __init__(self, rank: int, R: int, T_local: int, d: int, E: int, K: int, I: int,
                 weights: Dict[str, torch.Tensor], renorm: int = 1, device=None, kernels=None):
        if E % R:
            raise ValueError("R must divide E")
        self.k = kernels or CudaKernels()
        self.rank, self.R, self.T, self.d, self.E, self.K, self.I = rank, R, T_local, d, E, K, I
        self.El = E // R
        self.e_lo, self.e_hi = rank * self.El, (rank + 1) * self.El
        self.renorm = renorm
        dev = torch.device(device) if device is not None else weights["w_gate"].device
        self.device = dev
        self.w = weights
        self.shared = "ws_gate" in weights
        Tg = R * T_local
        self.Tg = Tg
        TK = Tg * K
        self.cap = Tg * min(K, self.El)
        cap = max(self.cap, 1)
        bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        # The local rows fill only the first offsets[e_hi] - offsets[e_lo] of the
        # capacity-sized row buffers, and the GEMMs see the whole capacity (the
        # count is known on the device only). The weight gradients multiply the
        # rows past the last local expert by zero rows in their straddling step,
        # so those rows must hold finite values: the row buffers and the backward
        # workspace start zeroed, and later steps leave only finite results there.
        z = lambda *s, dt: torch.zeros(*s, dtype=dt, device=dev)  # noqa: E731
        self.logits_all, self.x_all = e(Tg, E, dt=f32), e(Tg, d, dt=bf)
        self.topk_idx, self.topk_w = e(Tg, K, dt=i32), e(Tg, K, dt=f32)
        self.counts, self.offsets = e(E, dt=i32), e(E + 1, dt=i32)
        self.perm, self.inv_perm = e(TK, dt=i32), e(TK, dt=i32)
        self.xs, self.local_offsets = z(cap, d, dt=bf), e(self.El + 1, dt=i32)
        self.y, self.h, self.gu = z(cap, d, dt=bf), z(cap, I, dt=bf), z(cap, 2 * I, dt=bf)
        self.partial = e(Tg, d, dt=f32)
        self.out_partial = e(T_local, d, dt=f32)
        self.out = e(T_local, d, dt=bf)
        self.ws_perm = self.k.workspace(B.MOE_OP_BUILD_PERMUTATION, Tg, E, K, 1, 0, 0, dev)
        self.ws_ffn = self.k.workspace(B.MOE_OP_GROUPED_FFN, cap, self.El, 1, 1, d, I, dev)
        self.ws_bwd = self.k.workspace(B.MOE_OP_GROUPED_FFN_BACKWARD, cap, self.El, 1, 1, d, I, dev,
                                       zero=True)
        self.dout_all = e(Tg, d, dt=bf)
        self.dy, self.dxs = z(cap, d, dt=bf), z(cap, d, dt=bf)
        self.dtopk_w_partial, self.dtopk_w = e(Tg, K, dt=f32), e(T_local, K, dt=f32)
        self.dx_partial, self.dx_local_partial = e(Tg, d, dt=f32), e(T_local, d, dt=f32)
        self.dx, self.dlogits = e(T_local, d, dt=bf), e(T_local, E, dt=f32)
        El = self.El
        self.dw_gate, self.dw_up = e(El, d, I, dt=f32), e(El, d, I, dt=f32)
        self.dw_down = e(El, I, d, dt=f32)
        if self.shared:
            Is = weights["ws_gate"].shape[1]
            self.Is = Is
            self.ws_g, self.ws_u, self.ws_d = (weights[k].unsqueeze(0)
                                               for k in ("ws_gate", "ws_up", "ws_down"))
            self.s_offsets = torch.tensor([0, T_local], dtype=i32, device=dev)
            self.ys, self.hs, self.gus = e(T_local, d, dt=bf), e(T_local, Is, dt=bf), e(T_local, 2 * Is, dt=bf)
            self.dx_shared = e(T_local, d, dt=bf)
            self.dws_gate, self.dws_up = e(1, d, Is, dt=f32), e(1, d, Is, dt=f32)
            self.dws_down = e(1, Is, d, dt=f32)
            self.ws_sfwd = self.k.workspace(B.MOE_OP_GROUPED_FFN, T_local, 1, 1, 1, d, Is, dev)
            self.ws_sbwd = self.k.workspace(B.MOE_OP_GROUPED_FFN_BACKWARD, T_local, 1, 1, 1, d, Is,
                                            dev)

    def local_rows(self, t: torch.Tensor) -> torch.Tensor:
        return t[self.rank * self.T:(self.rank + 1) * self.T]

    def experts(self) -> None:
        """Replicated router on the gathered tokens, the local experts' rows, and
        the fp32 partial combine of every token."""
        k, w = self.k, self.w
        k.route_topk(self.logits_all, self.K, self.renorm, out=(self.topk_idx, self.topk_w))
        k.build_permutation(self.topk_idx, self.E, ws=self.ws_perm,
                            out=(self.counts, self.offsets, self.perm, self.inv_perm))
        k.dispatch_slice(self.x_all, self.inv_perm, self.offsets, self.K, self.e_lo, self.e_hi,
                         out=(self.xs, self.local_offsets))
        k.grouped_ffn(self.xs[:self.cap], self.local_offsets, w["w_gate"], w["w_up"], w["w_down"],
                      ws=self.ws_ffn, out=(self.y[:self.cap], self.h[:self.cap], self.gu[:self.cap]))
        k.combine_slice(self.y, self.topk_w, self.inv_perm, self.offsets, self.e_lo, self.e_hi,
                        out=self.partial)

    def finish(self, x_local: torch.Tensor) -> torch.Tensor:
        k = self.k
        self.x = x_local
        shared_y = None
        if self.shared:
            k.grouped_ffn(x_local, self.s_offsets, self.ws_g, self.ws_u, self.ws_d,
                          ws=self.ws_sfwd, out=(self.ys, self.hs, self.gus))
            shared_y = self.ys
        k.reduce_finish(self.out_partial, shared_y, out=self.out)
        return self.out

    def experts_backward(self) -> None:
        k, w, c = self.k, self.w, self.cap
        k.combine_backward_slice(self.dout_all, self.y, self.topk_w, self.inv_perm, self.offsets,
                                 self.e_lo, self.e_hi, out=(self.dy, self.dtopk_w_partial))
        k.grouped_ffn_backward_data(self.dy[:c], self.xs[:c], self.gu[:c], self.h[:c],
                                    self.local_offsets, w["w_gate"], w["w_up"], w["w_down"],
                                    ws=self.ws_bwd, out=self.dxs[:c])
        k.dispatch_backward_slice(self.dxs, self.inv_perm, self.offsets, self.Tg, self.K,
                                  self.e_lo, self.e_hi, out=self.dx_partial)
        k.grouped_ffn_backward_weights(self.dy[:c], self.xs[:c], self.h[:c], self.local_offsets,
                                       self.El, self.I, ws=self.ws_bwd,
                                       out=(self.dw_gate, self.dw_up, self.dw_down))

    def finish_backward(self, dout_local: torch.Tensor, logits_local: torch.Tensor) -> torch.Tensor:
        k = self.k
        dxs = None
        if self.shared:
            k.grouped_ffn_backward_data(dout_local, self.x, self.gus, self.hs, self.s_offsets,
                                        self.ws_g, self.ws_u, self.ws_d, ws=self.ws_sbwd,
                                        out=self.dx_shared)
            k.grouped_ffn_backward_weights(dout_local, self.x, self.hs, self.s_offsets, 1, self.Is,
                                           ws=self.ws_sbwd,
                                           out=(self.dws_gate, self.dws_up, self.dws_down))
            dxs = self.dx_shared
        k.reduce_finish(self.dx_local_partial, dxs, out=self.dx)
        k.route_topk_backward(None if self.renorm else logits_local,
                              self.local_rows(self.topk_idx), self.local_rows(self.topk_w),
                              self.dtopk_w, self.E, self.renorm, out=self.dlogits)
        return self.dx


def agrs_forward(ranks: Sequence[AGRSRank], ex: Exchange, logits: Sequence[torch.Tensor],
                 xs: Sequence[torch.Tensor]) -> List[torch.Tensor]:
    """Forward of all-gather / reduce-scatter EP: gather the group's logits and
    tokens, local experts on all of them, reduce-scatter the fp32 partials,
    add the shared expert and round on the owners."""
    ex.all_gather([rk.logits_all for rk in ranks], logits)
    ex.all_gather([rk.x_all for rk in ranks], xs)
    for rk in ranks:
        rk.experts()
    ex.reduce_scatter([rk.out_partial for rk in ranks], [rk.partial for rk in ranks])
    return [rk.finish(x) for rk, x in zip(ranks, xs)]


def agrs_backward(ranks: Sequence[AGRSRank], ex: Exchange, douts: Sequence[torch.Tensor],
                  logits: Sequence[torch.Tensor]) -> List[torch.Tensor]:
    """Backward: gather the upstream gradient, the local experts' backward,
    reduce-scatter the fp32 input gradient and the router-weight gradient,
    then the shared expert's and the router's backward on the owners."""
    ex.all_gather([rk.dout_all for rk in ranks], douts)
    for rk in ranks:
        rk.experts_backward()
    ex.reduce_scatter([rk.dx_local_partial for rk in ranks], [rk.dx_partial for rk in ranks])
    ex.reduce_scatter([rk.dtopk_w for rk in ranks], [rk.dtopk_w_partial for rk in ranks])
    return [rk.finish_backward(do, lg) for rk, do, lg in zip(ranks, douts, logits)]


def local_weights(weights: Dict[str, torch.Tensor], rank: int, R: int) -> Dict[str, torch.Tensor]:
    """The expert weights rank ``rank`` owns (contiguous blocks of E/R experts),
    plus the shared-expert weights unchanged."""
    E = weights["w_gate"].shape[0]
    El = E // R
    out = {k: weights[k][rank * El:(rank + 1) * El].contiguous() for k in ("w_gate", "w_up", "w_down")}
    for k in ("ws_gate", "ws_up", "ws_down"):
        if k in weights:
            out[k] = weights[k]
    return out


__all__ = ["Exchange", "ProcessGroupExchange", "LoopbackExchange", "CudaKernels", "A2ARank",
           "AGRSRank", "a2a_forward", "a2a_backward", "agrs_forward", "agrs_backward",
           "local_weights"]
