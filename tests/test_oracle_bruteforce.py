"""Brute force: every topk_idx in {-1..E-1}^(T*K) for one source of a tiny
R=2, E=4, K=2 set-up, the oracle against the independent dictionary-based
formulation in pyref.py."""
import itertools

import numpy as np
import pytest

import pyref

R, E, K = 2, 4, 2
L = E // R


def _cases(T):
    # source 0 takes every pattern; source 1 cycles through a few fixed ones
    others = [np.array(v, np.int64).reshape(T, K) for v in
              ([-1] * (T * K), list(range(T * K)), [3, 3, 0, -1, 1, 2][: T * K], [2, 1, 1, 2, 0, 0][: T * K])]
    others = [np.clip(o, -1, E - 1) for o in others]
    for i, combo in enumerate(itertools.product(range(-1, E), repeat=T * K)):
        idx = np.empty((R, T, K), np.int64)
        idx[0] = np.array(combo, np.int64).reshape(T, K)
        idx[1] = others[i % len(others)]
        yield idx


@pytest.mark.parametrize("T", [1, 2])
def test_layout_notify_dispatch_permute(orc, T):
    C = 2
    H = 8
    x = np.arange(R * T * H, dtype=np.uint16).reshape(R, T, H) + 1
    w = (np.arange(R * T * K, dtype=np.float32).reshape(R, T, K) + 1) / 16
    for idx in _cases(T):
        ref, valid = pyref.layout(idx, R, E, N=2)
        lay = orc.layout(idx, R, E, num_nodes=2)
        for key in ("num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank",
                    "num_tokens_per_node", "is_token_in_node"):
            np.testing.assert_array_equal(lay[key], ref[key], err_msg=f"{key} {idx.tolist()}")
        note = orc.notify(lay, R, E, T, C)
        sp, lists = pyref.send_pos(ref["is_token_in_rank"])
        # the offsets are relative to the receiver's block; rank_base locates the block
        for d in range(R):
            for i, (s, t) in enumerate(lists[d]):
                assert note["send_pos"][s, t, d] == i
            assert note["num_recv_tokens"][d] == len(lists[d])
        assert ((note["send_pos"] >= 0) == (sp >= 0)).all()
        np.testing.assert_array_equal(note["channel_prefix_matrix"],
                                      pyref.channel_prefix(ref["is_token_in_rank"], C))
        disp = orc.dispatch(x, idx, w, note, R, E)
        row = 0
        for d in range(R):
            for (s, t) in lists[d]:
                np.testing.assert_array_equal(disp["recv_x"][row], x[s, t])
                assert (disp["recv_src_rank"][row], disp["recv_src_idx"][row]) == (s, t)
                for k in range(K):
                    e = idx[s, t, k]
                    on_d = e >= 0 and e // L == d
                    assert disp["recv_topk_idx"][row, k] == (e - d * L if on_d else -1)
                    assert disp["recv_topk_weights"][row, k] == (w[s, t, k] if on_d else 0.0)
                row += 1
        perm = orc.permute(idx, disp["recv_x"], note, R, E)
        order, keys = pyref.permute_order(valid, R, E)
        assert perm["permuted_x"].shape[0] == len(keys) == int(note["perm_rank_base"][R])
        for (s, t, k), i in order.items():
            assert perm["perm_pos"][s, t, k] == i
            np.testing.assert_array_equal(perm["permuted_x"][i], x[s, t])
        assert (perm["perm_pos"] >= 0).sum() == len(order)


@pytest.mark.parametrize("T", [1, 2])
def test_low_latency_slots(orc, T):
    H = 128
    cap = 4  # a source sends at most T*K = 4 entries to one expert
    x = np.zeros((R, T, H), np.uint16)
    for idx in _cases(T):
        _, valid = pyref.layout(idx, R, E)
        sent = orc.ll_send(x, idx, R, E, cap)
        slot, counts = pyref.ll_slots(valid, R, E, T, K, 0, T)
        for s in range(R):
            for e in range(E):
                assert sent["counts"][e, s] == counts.get((s, e), 0)
            for t in range(T):
                for k in range(K):
                    assert sent["slot"][s, t, k] == slot.get((s, t, k), -1)
        # every valid entry's region address is distinct and inside the buffer
        addrs = [((idx[s, t, k] * R + s) * cap + slot[(s, t, k)]) for (s, t, k) in valid]
        assert len(set(addrs)) == len(addrs)
        assert all(0 <= a < E * R * cap for a in addrs)
        for (s, t, k) in valid:
            a = (idx[s, t, k] * R + s) * cap + slot[(s, t, k)]
            assert sent["reg_src"][a] == t


@pytest.mark.parametrize("T", [1, 2])
def test_hier_stage_positions(orc, T):
    N = 2
    for idx in _cases(T):
        ref, _ = pyref.layout(idx, R, E, N=N)
        lay = orc.layout(idx, R, E, num_nodes=N)
        base, pos = orc.hier_stage_pos(lay, R, T, N)
        rpos, rbase = pyref.stage_positions(ref["is_token_in_node"], R, N)
        np.testing.assert_array_equal(base, rbase)
        for s in range(R):
            for t in range(T):
                for n in range(N):
                    assert pos[s, t, n] == rpos.get((s, t, n), -1)


def test_combine_exact_small(orc):
    """ord32 and the hierarchical order against an exact-arithmetic restatement
    (fp32 fma per rank, ranks summed ascending; for the hierarchical order the
    rank partials of a node summed first, then the nodes ascending) on random
    tiny cases with 4 ranks and 2 nodes, values over a wide dynamic range so
    that the order of three or more partials changes the rounding, including
    tokens with several experts on one rank."""
    import torch
    rng = np.random.default_rng(3)
    R4, E4, K4, N4 = 4, 8, 4, 2
    L4, G4 = E4 // R4, R4 // N4
    T, H = 3, 8
    for trial in range(40):
        idx = rng.integers(-1, E4, size=(R4, T, K4)).astype(np.int64)
        xw = (rng.standard_normal((R4, T, H)) * np.exp(rng.uniform(-6, 6, (R4, T, H)))).astype(np.float32)
        x = torch.from_numpy(xw).to(torch.bfloat16)
        xb = x.view(torch.int16).numpy().view(np.uint16)
        w = (rng.standard_normal((R4, T, K4)) * np.exp(rng.uniform(-4, 4, (R4, T, K4)))).astype(np.float32)
        lay = orc.layout(idx, R4, E4)
        note = orc.notify(lay, R4, E4, T, 2)
        disp = orc.dispatch(x, idx, w, note, R4, E4)
        perm = orc.permute(idx, disp["recv_x"], note, R4, E4)
        out = orc.combine(perm["permuted_x"], perm["perm_pos"], idx, w, R4, E4, "ord32")
        hout = orc.combine_hier(perm["permuted_x"], perm["perm_pos"], idx, w, R4, E4, N4)
        for s in range(R4):
            for t in range(T):
                for j in range(H):
                    xv = pyref.bf16_value(xb[s, t, j])
                    partial = {}
                    for d in range(R4):
                        ks = [k for k in range(K4) if idx[s, t, k] >= 0 and idx[s, t, k] // L4 == d]
                        if not ks:
                            continue
                        p = 0.0
                        for k in ks:
                            p = pyref.fmaf(float(w[s, t, k]), xv, p)
                        partial[d] = p
                    final = 0.0
                    for d in sorted(partial):
                        final = pyref.fadd(final, partial[d])
                    assert out[s, t, j] == pyref.bf16_bits_of(final), (trial, s, t, j)
                    hfinal = 0.0
                    for n in range(N4):
                        ds = [d for d in sorted(partial) if d // G4 == n]
                        if not ds:
                            continue
                        node = 0.0
                        for d in ds:
                            node = pyref.fadd(node, partial[d])
                        hfinal = pyref.fadd(hfinal, node)
                    assert hout[s, t, j] == pyref.bf16_bits_of(hfinal), (trial, s, t, j)
