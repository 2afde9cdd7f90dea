"""Randomised configurations (a fixed list of seeds): sizes, channel counts,
nodes, masks, duplicate experts, expert alignment and low-latency
microbatches drawn at random, every result compared with the oracle bit for
bit (the normal path through compare_normal, which also checks the fused
dispatch; the low-latency path slot by slot)."""
import numpy as np
import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, LLBuffer, inputs
from parity_util import bits, compare_normal, eq

pytestmark = pytest.mark.gpu

SEEDS = list(range(100, 124))


def _draw(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
    L = int(rng.choice([1, 2, 3, 4, 8, 16]))
    E = R * L
    K = int(rng.integers(1, min(E, 9) + 1))
    T = int(rng.choice([0, 1, 7, 33, 256, 257, 300]))
    H = int(rng.choice([8, 64, 136, 256, 512]))
    C = int(rng.integers(1, 9))
    divisors = [n for n in range(1, R + 1) if R % n == 0]
    N = int(rng.choice(divisors))
    mask_p = float(rng.choice([0.0, 0.0, 0.1, 0.5]))
    distinct = bool(rng.random() < 0.8)
    return R, E, K, T, H, C, N, mask_p, distinct


@pytest.mark.parametrize("seed", SEEDS)
def test_normal_random_config(seed):
    R, E, K, T, H, C, N, mask_p, distinct = _draw(seed)
    idx = inputs.random_topk(R, E, K, T, seed, mask_p, distinct)
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    compare_normal(R, E, K, T, H, C, x, idx, w, nodes=N, hier=N > 1)


@pytest.mark.parametrize("seed", SEEDS[:12])
def test_aligned_random_config(seed):
    R, E, K, T, H, C, N, mask_p, distinct = _draw(seed)
    align = int(np.random.default_rng(seed + 1).choice([2, 8, 64]))
    idx = inputs.random_topk(R, E, K, T, seed, mask_p, distinct)
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    ctx = Context(R, E, K, T, H, num_channels=C, expert_alignment=align)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    lay, h = ctx.layout_notify(idxd)
    perm = ctx.permute(h, ctx.dispatch(xd, idxd, wd, h))
    out = ctx.combine(h, perm["permuted_x"], idxd, wd)
    ctx.check()
    o_note = orc.notify(orc.layout(idx, R, E), R, E, T, C, align=align)
    eq(h["expert_offsets"], o_note["expert_offsets"], "expert_offsets")
    o_disp = orc.dispatch(x, idx, w, o_note, R, E)
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    eq(h["perm_pos"], o_perm["perm_pos"], "perm_pos")
    used = o_perm["perm_src_row"] >= 0
    eq(bits(perm["permuted_x"])[used], o_perm["permuted_x"][used], "permuted_x")
    eq(out, orc.combine(o_perm["permuted_x"], o_perm["perm_pos"], idx, w, R, E, "ord32"), "combine")


@pytest.mark.parametrize("seed", SEEDS[:16])
def test_low_latency_random_config(seed):
    rng = np.random.default_rng(seed + 7)
    R = int(rng.choice([1, 2, 4, 8, 16]))
    E = R * int(rng.choice([1, 2, 4, 8]))
    K = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.choice([1, 5, 40, 96]))
    H = int(rng.choice([128, 256, 1024]))
    cap = int(rng.integers(1, T + 1))
    idx = inputs.random_topk(R, E, K, T, seed, float(rng.choice([0.0, 0.2])))
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    buf = LLBuffer(R, E, K, T, H, cap)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    out = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
    o_out = np.zeros((R, T, H), np.uint16)
    out_r = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
    o_out_r = np.zeros((R, T, H), np.uint16)
    L = E // R
    yr = inputs.random_rows(R * L * R * cap, H, seed=seed).view(R, L, R * cap, H)
    yrd = yr.cuda()
    for t0 in range(0, T, cap):
        n = min(cap, T - t0)
        pk = buf.dispatch(xd, idxd, t0, n)
        sent = orc.ll_send(x, idx, R, E, cap, t0, n)
        o_pk = orc.ll_pack(sent, R, E, H, cap)
        eq(pk["slot"][:, t0:t0 + n], sent["slot"][:, t0:t0 + n], "slot")
        eq(pk["packed_recv_count"], o_pk["packed_recv_count"], "packed_recv_count")
        eq(pk["layout_range"], o_pk["layout_range"], "layout_range")
        px, ps = bits(pk["packed_x"]), bits(pk["packed_scales"])
        for d in range(R):
            for l in range(L):
                c = int(o_pk["packed_recv_count"][d, l])
                eq(px[d, l, :c], o_pk["packed_x"][d, l, :c], "packed_x")
                eq(ps[d, l, :c], o_pk["packed_scales"][d, l, :c], "packed_scales")
        y = orc.ll_dequant(o_pk["packed_x"], o_pk["packed_scales"])
        buf.combine(torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda(), idxd, wd, pk, t0, n, out=out)
        orc.ll_combine(y, idx, w, sent["slot"], o_pk["layout_range"], R, E, cap, t0, n, out=o_out)
        buf.combine(yrd, idxd, wd, pk, t0, n, out=out_r)
        orc.ll_combine(yr, idx, w, sent["slot"], o_pk["layout_range"], R, E, cap, t0, n, out=o_out_r)
    buf.check()
    eq(out, o_out, "ll combine")
    eq(out_r, o_out_r, "ll combine of distinct expert rows")


def _wide_range_x(R, T, H, seed):
    """bf16 rows whose 128-channel blocks span magnitudes from 2^-40 to 2^40
    (power-of-two scalings of N(0,1), exact in bf16 above the subnormal range),
    with some all-zero blocks, so that the FP8 scales cover many binades."""
    x = inputs.random_x(R, T, H, seed).float()
    rng = np.random.default_rng(seed + 11)
    nb = H // 128
    e = rng.integers(-40, 41, size=(R, T, nb)).astype(np.float64)
    scale = np.exp2(e)
    scale[rng.random((R, T, nb)) < 0.05] = 0.0
    s = torch.from_numpy(np.repeat(scale, 128, axis=2)).float()
    return (x * s).to(torch.bfloat16)


@pytest.mark.parametrize("seed", SEEDS[:12])
def test_fp8_random_config(seed):
    """The FP8 rows from the quantiser, the one-pass dispatch into the permuted
    layout and the one-pass dispatch into the receive layout, on random
    configurations with block maxima over many binades, against the oracle's
    quantiser row by row."""
    rng = np.random.default_rng(seed + 3)
    R = int(rng.choice([1, 2, 4, 8]))
    E = R * int(rng.choice([1, 2, 4, 8]))
    K = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.choice([1, 7, 33, 130]))
    H = int(rng.choice([128, 256, 384, 1024, 2048]))
    C = int(rng.integers(1, 5))
    mask_p = float(rng.choice([0.0, 0.1]))
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    x = _wide_range_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    ctx = Context(R, E, K, T, H, num_channels=C)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    h = ctx.notify_dispatch(idxd, ctx.get_dispatch_layout(idxd))
    n_def = H + H // 32
    xb = bits(x).reshape(R * T, H)
    o_rows = np.zeros((R * T, n_def), np.uint8)
    for g in range(R * T):
        codes, scales = orc.quantize_row(xb[g])
        o_rows[g, :H] = codes
        o_rows[g, H:] = scales.view(np.uint8)
    xq = ctx.quantize_fp8(xd)
    perm = ctx.dispatch_permuted_quant(xd, idxd, wd, h)
    recv = ctx.dispatch_quant(xd, idxd, wd, h)
    ctx.check()
    eq(bits(xq)[:, :n_def], o_rows, "quantised rows")
    pp = h["perm_pos"].cpu().numpy().reshape(R * T, K)
    got = bits(perm["permuted_xq"])
    for g, k in zip(*np.nonzero(pp >= 0)):
        eq(got[pp[g, k], :n_def], o_rows[g], f"permuted row of token {g}, entry {k}")
    sp = h["send_pos"].cpu().numpy().reshape(R * T, R)
    rb = h["rank_base"].cpu().numpy()
    gr = bits(recv["recv_xq"])
    for g, d in zip(*np.nonzero(sp >= 0)):
        eq(gr[rb[d] + sp[g, d], :n_def], o_rows[g], f"received row of token {g} at rank {d}")
