"""CPU stand-ins for the per-rank steps of the expert-parallel layers, for the
multi-process tests over gloo (no GPU). Each method has the signature of the
library call it replaces and writes its results into the given CPU tensors;
the arithmetic is the oracle's (float64, the same bf16 rounding points).

Test infrastructure only: the package's EP classes take these through their
``kernels`` argument; the package itself has no CPU path."""
import numpy as np
import torch

from oracle import moe_oracle as O


def _f64(t):
    return t.detach().to(torch.float64).numpy()


def _put(dst, arr):
    dst.copy_(torch.from_numpy(np.ascontiguousarray(arr)).to(dst.dtype))


class CpuKernels:
    def __init__(self):
        self._stash = {}

    def workspace(self, op, T, E, K, R, d, I, device, zero=False):
        return torch.zeros(1, dtype=torch.uint8)

    def route_topk(self, logits, K, renorm=1, out=None):
        idx, w = O.route_topk(_f64(logits), K, renorm)
        _put(out[0], idx)
        _put(out[1], w)
        return out

    def route_topk_backward(self, logits, topk_idx, topk_w, dtopk_w, E, renorm=1, out=None):
        T = topk_idx.shape[0]
        lg = _f64(logits) if logits is not None else np.zeros((T, E))
        _put(out, O.route_topk_backward(lg, topk_idx.numpy(), _f64(topk_w), _f64(dtopk_w), renorm))
        return out

    def build_permutation(self, topk_idx, E, ws=None, out=None):
        idx = topk_idx.numpy()
        counts, offsets = O.expert_counts_offsets(idx, E)
        perm, inv = O.stable_permutation(idx, E)
        for dst, a in zip(out, (counts, offsets, perm, inv)):
            _put(dst, a)
        return out

    def dispatch(self, x, perm, K, out=None):
        _put(out, O.dispatch(_f64(x), perm.numpy(), K))
        return out

    def dispatch_scatter(self, x, inv_perm, K, out=None):
        xv = _f64(x)
        ip = inv_perm.numpy().astype(np.int64)
        res = np.zeros((ip.size, xv.shape[1]))
        res[ip] = xv[np.arange(ip.size) // K]
        _put(out, res)
        return out

    def ep_recv_layout(self, counts_local, recv_counts, R, capacity, host_splits=None, ws=None,
                       out=None):
        """Splits, local offsets and regroup index written out by their definition:
        the receive buffer is source-major, each source's block expert-major; the
        regrouped order is (local expert, source, the source's order)."""
        E = counts_local.numel()
        El = E // R
        c = counts_local.numpy().astype(np.int64)
        C = recv_counts.numpy().astype(np.int64).reshape(R, El)
        send = [int(c[q * El:(q + 1) * El].sum()) for q in range(R)]
        recv = [int(C[s].sum()) for s in range(R)]
        splits, loff, reg = out
        _put(splits, np.array(send + recv))
        if host_splits is not None:
            _put(host_splits, np.array(send + recv))
        # receive-buffer row of (source s, local expert e, i-th row)
        rows = {}
        pos = 0
        for s in range(R):
            for e in range(El):
                for i in range(C[s, e]):
                    rows[(s, e, i)] = pos
                    pos += 1
        order = [rows[(s, e, i)] for e in range(El) for s in range(R) for i in range(C[s, e])]
        offs = [0]
        for e in range(El):
            offs.append(offs[-1] + int(C[:, e].sum()))
        _put(loff, np.array(offs))
        if order:
            _put(reg[:len(order)], np.array(order))
        return out

    # grouped FFN: forward in one call, backward data part computes everything
    def grouped_ffn(self, xp, offsets, w_gate, w_up, w_down, ws=None, out=None):
        y, h, gu = out
        M = xp.shape[0]
        off = offsets.numpy().astype(np.int64)
        if M == 0 or off[-1] == 0:
            return out
        n = int(off[-1])
        yy, gg, hh = O.grouped_ffn(_f64(xp)[:n], off, _f64(w_gate), _f64(w_up), _f64(w_down))
        _put(y[:n], yy)
        _put(gu[:n], gg)
        _put(h[:n], hh)
        return out

    def grouped_ffn_backward_data(self, dy, xp, gu, h, offsets, w_gate, w_up, w_down, ws=None,
                                  out=None):
        off = offsets.numpy().astype(np.int64)
        n = int(off[-1])
        E, d, I = w_gate.shape
        if n == 0:
            self._stash[id(ws)] = (np.zeros((E, d, I)), np.zeros((E, d, I)), np.zeros((E, I, d)))
            return out
        dxp, dwg, dwu, dwd = O.grouped_ffn_backward(_f64(dy)[:n], _f64(xp)[:n], _f64(gu)[:n],
                                                    _f64(h)[:n], off, _f64(w_gate), _f64(w_up),
                                                    _f64(w_down))
        _put(out[:n], dxp)
        self._stash[id(ws)] = (dwg, dwu, dwd)
        return out

    def grouped_ffn_backward_weights(self, dy, xp, h, offsets, E, I, ws=None, out=None):
        for dst, a in zip(out, self._stash.pop(id(ws))):
            _put(dst, a)
        return out

    def combine(self, y, topk_w, inv_perm, shared_y=None, out=None):
        K = topk_w.shape[1]
        sy = _f64(shared_y) if shared_y is not None else None
        _put(out, O.combine(_f64(y), _f64(topk_w), inv_perm.numpy(), K, sy))
        return out

    def combine_backward(self, dout, y, topk_w, inv_perm, out=None):
        K = topk_w.shape[1]
        dy, dw = O.combine_backward(_f64(dout), _f64(y), _f64(topk_w), inv_perm.numpy(), K)
        _put(out[0], dy)
        _put(out[1], dw)
        return out

    def dispatch_backward(self, dxp, inv_perm, T, K, dx_shared=None, out=None):
        ds = _f64(dx_shared) if dx_shared is not None else None
        _put(out, O.dispatch_backward(_f64(dxp), inv_perm.numpy(), K, T, ds))
        return out

    # all-gather / reduce-scatter slices
    @staticmethod
    def _window(offsets, e_lo, e_hi):
        off = offsets.numpy()
        return int(off[e_lo]), int(off[e_hi])

    def dispatch_slice(self, x, inv_perm, offsets, K, e_lo, e_hi, out=None):
        lo, hi = self._window(offsets, e_lo, e_hi)
        xs, loff = out
        ip = inv_perm.numpy().astype(np.int64)
        xv = _f64(x)
        for a, p in enumerate(ip):
            if lo <= p < hi:
                _put(xs[p - lo], xv[a // K])
        _put(loff, offsets.numpy()[e_lo:e_hi + 1] - lo)
        return out

    def combine_slice(self, y_local, topk_w, inv_perm, offsets, e_lo, e_hi, out=None):
        lo, hi = self._window(offsets, e_lo, e_hi)
        T, K = topk_w.shape
        ip = inv_perm.numpy().astype(np.int64).reshape(T, K)
        w = _f64(topk_w)
        yv = _f64(y_local)
        acc = np.zeros((T, yv.shape[1]))
        for t in range(T):
            for j in range(K):
                if lo <= ip[t, j] < hi:
                    acc[t] += w[t, j] * yv[ip[t, j] - lo]
        _put(out, acc)
        return out

    def combine_backward_slice(self, dout, y_local, topk_w, inv_perm, offsets, e_lo, e_hi,
                               out=None):
        lo, hi = self._window(offsets, e_lo, e_hi)
        T, K = topk_w.shape
        ip = inv_perm.numpy().astype(np.int64).reshape(T, K)
        w, do, yv = _f64(topk_w), _f64(dout), _f64(y_local)
        dy, dw = out
        dwv = np.zeros((T, K))
        for t in range(T):
            for j in range(K):
                p = ip[t, j]
                if lo <= p < hi:
                    _put(dy[p - lo], O.round_bf16(w[t, j] * do[t]))
                    dwv[t, j] = do[t] @ yv[p - lo]
        _put(dw, dwv)
        return out

    def dispatch_backward_slice(self, dxs, inv_perm, offsets, T, K, e_lo, e_hi, out=None):
        lo, hi = self._window(offsets, e_lo, e_hi)
        ip = inv_perm.numpy().astype(np.int64).reshape(T, K)
        dv = _f64(dxs)
        acc = np.zeros((T, dv.shape[1]))
        for t in range(T):
            for j in range(K):
                if lo <= ip[t, j] < hi:
                    acc[t] += dv[ip[t, j] - lo]
        _put(out, acc)
        return out

    def reduce_finish(self, partial, extra=None, out=None):
        acc = _f64(partial)
        if extra is not None:
            acc = acc + _f64(extra)
        _put(out, O.round_bf16(acc))
        return out
