"""Pins of the oracle's histogram, stable permutation and simulated EP layout.

Pins: invariants the pages state (counts sum to T*K, the packing is a bijection
grouped by expert, every rank receives exactly the tokens routed to its expert
slice, the receive buffer is source-major), the pages' own per-expert loop,
exhaustive enumeration, a python-level simulation of the all-to-all, and a
hand-derived worked example.
"""
import itertools
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            if not ln.strip() or ln.startswith("#"):
                continue
            k, *v = ln.split()
            vals[k] = np.array([int(x) for x in v], dtype=np.int64)
    return vals


def test_golden_pack_example():
    g = _read_golden("pack_example.txt")
    T, K, E, R = (int(g[k][0]) for k in ("T", "K", "E", "R"))
    idx = g["topk_idx"].reshape(T, K)
    counts, offsets = O.expert_counts_offsets(idx, E)
    perm, inv = O.stable_permutation(idx, E)
    assert np.array_equal(counts, g["counts"])
    assert np.array_equal(offsets, g["offsets"])
    assert np.array_equal(perm, g["perm"])
    assert np.array_equal(inv, g["inv_perm"])
    ep = O.ep_layout(idx, T, E, K, R)
    assert np.array_equal(ep["ep_counts"].reshape(-1), g["ep_counts"])
    assert np.array_equal(ep["send_splits"].reshape(-1), g["send_splits"])
    for k in ("send_index", "a2a_index", "regroup_index"):
        assert np.array_equal(ep[k], g[k]), k


def _random_idx(rng, T, E, K):
    # distinct experts per token, like a top-k
    return np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)


def _check_perm_invariants(idx, E):
    T, K = idx.shape
    flat = idx.reshape(-1)
    counts, offsets = O.expert_counts_offsets(idx, E)
    perm, inv = O.stable_permutation(idx, E)
    assert counts.sum() == T * K and offsets[-1] == T * K and offsets[0] == 0
    assert (np.diff(offsets) == counts).all()
    assert np.array_equal(np.sort(perm), np.arange(T * K))           # bijection
    assert np.array_equal(inv[perm], np.arange(T * K))
    assert (np.diff(flat[perm]) >= 0).all()                           # grouped
    for e in range(E):                                                # stable
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()
        assert (flat[seg] == e).all()
    assert np.array_equal(perm, O.permutation_by_expert_loop(idx, E))  # pages' loop
    return counts, offsets, perm, inv


def test_permutation_invariants_random():
    rng = np.random.default_rng(0)
    for (T, E, K) in [(1, 1, 1), (5, 4, 2), (64, 8, 2), (257, 16, 3), (200, 128, 8)]:
        idx = _random_idx(rng, T, E, K)
        counts, *_ = _check_perm_invariants(idx, E)
        assert (counts <= T).all()


def test_permutation_exhaustive_small():
    # every expert assignment of TK <= 8 slots over E <= 4 experts
    for E, TK in [(2, 8), (3, 6), (4, 6)]:
        allv = np.array(list(itertools.product(range(E), repeat=TK)), dtype=np.int32)
        for row in allv:
            idx = row.reshape(TK, 1)
            perm, inv = O.stable_permutation(idx, E)
            ref = sorted(range(TK), key=lambda a: (int(row[a]), a))
            assert list(perm) == ref


def _simulate_all_to_all(idx, T, E, K, R):
    """Message-level simulation with python lists: what each rank packs, what it
    sends to each rank, what each rank receives and how it regroups."""
    El = E // R
    flat = [int(v) for v in idx.reshape(-1)]
    per = T // R
    send_bufs = []
    for s in range(R):
        mine = [a for a in range(s * per * K, (s + 1) * per * K)]
        packed = []
        for e in range(E):                     # expert-major packing on the sender
            packed += [a for a in mine if flat[a] == e]
        send_bufs.append(packed)
    send_flat = [a for buf in send_bufs for a in buf]
    recv = []
    for d in range(R):
        buf = []
        for s in range(R):                      # source-major receive
            buf += [a for a in send_bufs[s] if flat[a] // El == d]
        recv.append(buf)
    recv_flat = [a for buf in recv for a in buf]
    grouped = []
    for d in range(R):
        for el in range(El):                    # local-expert-major regroup
            grouped += [a for a in recv[d] if flat[a] == d * El + el]
    return send_flat, recv_flat, grouped, send_bufs, recv


@pytest.mark.parametrize("T,E,K,R", [(4, 4, 2, 2), (8, 8, 2, 4), (12, 6, 3, 3), (16, 8, 4, 1),
                                     (32, 16, 4, 4), (64, 8, 2, 2)])
def test_ep_layout_against_simulation(T, E, K, R):
    rng = np.random.default_rng(T * 100 + E)
    for trial in range(5):
        idx = _random_idx(rng, T, E, K)
        ep = O.ep_layout(idx, T, E, K, R)
        send_flat, recv_flat, grouped, send_bufs, recv = _simulate_all_to_all(idx, T, E, K, R)
        send = ep["send_index"]
        a2a = ep["a2a_index"]
        reg = ep["regroup_index"]
        assert list(send) == send_flat
        assert [int(send[q]) for q in a2a] == recv_flat
        assert [recv_flat[r] for r in reg] == grouped
        # split matrices
        El = E // R
        for s in range(R):
            for d in range(R):
                n = sum(1 for a in send_bufs[s] if int(idx.reshape(-1)[a]) // El == d)
                assert ep["send_splits"][s, d] == n


@pytest.mark.parametrize("T,E,K,R", [(64, 8, 2, 2), (96, 16, 4, 4), (64, 16, 3, 8), (40, 8, 2, 1)])
def test_ep_layout_invariants(T, E, K, R):
    rng = np.random.default_rng(7)
    idx = _random_idx(rng, T, E, K)
    flat = idx.reshape(-1)
    El = E // R
    counts, offsets = O.expert_counts_offsets(idx, E)
    perm, _ = O.stable_permutation(idx, E)
    ep = O.ep_layout(idx, T, E, K, R)
    C, S = ep["ep_counts"], ep["send_splits"]
    assert C.sum() == T * K and S.sum() == T * K
    assert np.array_equal(C.sum(axis=0), counts)
    assert (C.sum(axis=1) == T * K // R).all()
    # composition: send -> exchange -> regroup reproduces the packing
    assert np.array_equal(ep["send_index"][ep["a2a_index"][ep["regroup_index"]]], perm)
    assert np.array_equal(ep["group_order"], perm)
    # each destination's receive range holds exactly the assignments for its experts,
    # laid out by source rank with block sizes S[s, d]
    recv_a = ep["send_index"][ep["a2a_index"]]
    r0 = 0
    for d in range(R):
        n_d = int(S[:, d].sum())
        blk = recv_a[r0:r0 + n_d]
        assert set(blk.tolist()) == set(np.nonzero(flat // El == d)[0].tolist())
        src = (blk // K) // (T // R)
        assert (np.diff(src) >= 0).all()
        assert np.array_equal(np.bincount(src, minlength=R), S[:, d])
        r0 += n_d
    if R == 1:
        assert np.array_equal(ep["regroup_index"], np.arange(T * K))
        assert np.array_equal(ep["a2a_index"], np.arange(T * K))
        assert np.array_equal(ep["send_index"], perm)
