"""Pins of the oracle's low-latency dequantisation and combine and of its
hierarchical staging (stage A into the home rank, stage B forwarded to the
ranks of the node), each against something other than the oracle itself.

* LL combine ([P1] 低延迟模式: the combine stays BF16; the sum runs over the
  token's top-k entries in k order, fp32 fused multiply-add):
  - exact: pyref's dictionary-based packed positions and exact rational fma
    on y rows with a distinct, wide-range value per packed row and channel,
    so that reading any other row (another k of the same token included)
    changes the bits;
  - closed forms: partials 2^25, -2^25, 1 placed so that k order and rank
    order give different bf16 results; a product whose fp32 rounding
    residual survives only under a fused multiply-add.
* LL dequantisation (y = bf16(fp32(e4m3 value * scale))): every code against
  torch.float8_e4m3fn's decode times the block's scale, with a different
  scale in every 128-channel block.
* Hierarchical staging ([P2] hybrid 模式; [P1] 零拷贝通信, home rank on the
  target node): staged rows against pyref's (home rank, s, t) enumeration,
  forwarded rows against pyref's (s, t) receive lists, and the staged
  recv_x equal to the flat dispatch's recv_x (worked case and random cases).
"""
import numpy as np
import pytest
import torch

import pyref
from combine_get_dispatch_histograms_gb300 import inputs
from golden_io import load


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _wide_bf16(shape, rng):
    """bf16 values with a random sign, 7 random mantissa bits and exponents
    over [-30, 30]: every value distinct with high probability."""
    sign = rng.choice([-1.0, 1.0], size=shape)
    mant = 1.0 + rng.integers(0, 128, size=shape) / 128.0
    ex = rng.integers(-30, 31, size=shape).astype(np.float64)
    return torch.from_numpy(sign * mant * np.exp2(ex)).to(torch.bfloat16)


def _ll_inputs(R, E, K, T, cap, t0, n, seed, mask_p, distinct=True):
    idx = inputs.random_topk(R, E, K, T, seed, mask_p, distinct).numpy()
    rng = np.random.default_rng(seed)
    # weights over several binades, both signs
    w = (rng.choice([-1.0, 1.0], size=(R, T, K)) * rng.random((R, T, K)) *
         np.exp2(rng.integers(-6, 7, size=(R, T, K)))).astype(np.float32)
    _, valid = pyref.layout(idx, R, E)
    where = pyref.ll_packed_rows(valid, R, E, T, K, t0, n)
    return idx, w, valid, where


def _layout_range_and_slot(valid, where, R, E, T, K, t0, n):
    """The packed layout's (begin, count) per (d, l, s) and the slot per
    (s, t, k), from pyref's enumeration (not from the oracle's send/pack)."""
    L = E // R
    slot_d, counts = pyref.ll_slots(valid, R, E, T, K, t0, n)
    lr = np.zeros((R, L, R, 2), np.int32)
    for e in range(E):
        d, l = divmod(e, L)
        begin = 0
        for s in range(R):
            c = counts.get((s, e), 0)
            lr[d, l, s] = (begin, c)
            begin += c
    slot = np.full((R, T, K), -1, np.int32)
    for key, i in slot_d.items():
        slot[key] = i
    return lr, slot


@pytest.mark.parametrize("R,E,K,T,cap,t0,n,mask_p,distinct,seed", [
    (2, 4, 3, 3, 3, 0, 3, 0.0, True, 0),
    (4, 8, 2, 5, 3, 2, 3, 0.2, True, 1),     # a microbatch in the middle, masks
    (2, 4, 3, 4, 4, 0, 4, 0.0, False, 2),    # duplicate experts inside a token
])
def test_ll_combine_exact(orc, R, E, K, T, cap, t0, n, mask_p, distinct, seed):
    H = 8
    idx, w, valid, where = _ll_inputs(R, E, K, T, cap, t0, n, seed, mask_p, distinct)
    L = E // R
    # duplicates can put more than cap entries of one source into one region:
    # size the regions for the largest count
    _, counts = pyref.ll_slots(valid, R, E, T, K, t0, n)
    cap = max([cap] + list(counts.values()))
    lr, slot = _layout_range_and_slot(valid, where, R, E, T, K, t0, n)
    rng = np.random.default_rng(100 + seed)
    y = _wide_bf16((R, L, R * cap, H), rng)
    yb = _bits(y)
    y_rows = {(d, l, r): [pyref.bf16_value(b) for b in yb[d, l, r]]
              for d in range(R) for l in range(L) for r in range(R * cap)}
    exp = pyref.ll_combine_exact(y_rows, where, idx, w, t0, n)
    got = orc.ll_combine(y, idx, w, slot, lr, R, E, cap, t0, n)
    for (s, t), vals in exp.items():
        np.testing.assert_array_equal(got[s, t], np.array(vals, np.uint16), err_msg=f"token ({s}, {t})")
    # tokens outside the microbatch are left as they were (zero)
    outside = [t for t in range(T) if not t0 <= t < t0 + n]
    assert (got[:, outside] == 0).all()


def _ll_closed_form(orc, experts, weights, yvals):
    """One token (s=0, t=0) of R=4, E=8 (expert e on rank e // 2) with the
    given experts, weights and one y value per entry (all channels)."""
    R, E, K, T, H, cap = 4, 8, len(experts), 1, 8, 1
    idx = np.full((R, T, K), -1, np.int64)
    idx[0, 0] = experts
    w = np.zeros((R, T, K), np.float32)
    w[0, 0] = weights
    _, valid = pyref.layout(idx, R, E)
    where = pyref.ll_packed_rows(valid, R, E, T, K, 0, 1)
    lr, slot = _layout_range_and_slot(valid, where, R, E, T, K, 0, 1)
    y = torch.zeros(R, E // R, R * cap, H, dtype=torch.float32)
    for k in range(K):
        y[where[(0, 0, k)]] = yvals[k]
    return orc.ll_combine(y.to(torch.bfloat16), idx, w, slot, lr, R, E, cap)[0, 0]


def test_ll_combine_sums_in_k_order_not_rank_order(orc):
    big = float(2 ** 25)
    # k = 0, 1, 2 on ranks 3, 1, 0: k order (2^25 - 2^25) + 1 = 1; rank order
    # (1 - 2^25) + 2^25 = 0, since fp32 spacing at 2^25 is 4 and the 1 is lost
    out = _ll_closed_form(orc, [6, 2, 0], [1.0, 1.0, 1.0], [big, -big, 1.0])
    assert (out == pyref.bf16_bits_of(1.0)).all()
    # the reverse k order gives the rank-order result
    out = _ll_closed_form(orc, [0, 2, 6], [1.0, 1.0, 1.0], [1.0, -big, big])
    assert (out == pyref.bf16_bits_of(0.0)).all()


def test_ll_combine_is_a_fused_multiply_add_chain(orc):
    # acc = w0 * 1 = -(1 + 2^-7 + 2^-17) exactly; then w1 * y1 with
    # w1 = 1 + 2^-17, y1 = 1 + 2^-7 (a bf16 value): the exact product is
    # 1 + 2^-7 + 2^-17 + 2^-24, a tie in fp32 that rounds to even (dropping
    # 2^-24).  Fused: 2^-24 survives; multiply then add: 0.
    w0 = -(1.0 + 2.0 ** -7 + 2.0 ** -17)
    w1 = 1.0 + 2.0 ** -17
    assert float(np.float32(w0)) == w0 and float(np.float32(w1)) == w1
    out = _ll_closed_form(orc, [0, 1], [w0, w1], [1.0, 1.0 + 2.0 ** -7])
    assert (out == pyref.bf16_bits_of(2.0 ** -24)).all()
    assert pyref.bf16_bits_of(2.0 ** -24) != 0


def test_ll_dequant_every_code_with_block_distinct_scales(orc):
    rows, H = 8, 512  # 32 blocks of 128 channels
    S = H // 128
    rng = np.random.default_rng(3)
    codes = np.empty((rows, H), np.uint8)
    for r in range(rows):
        for b in range(S):
            codes[r, b * 128:(b + 1) * 128] = ((r * S + b) % 2) * 128 + rng.permutation(128)
    # scales: 1, 0, powers of two, and random fp32 values over a wide range
    scales = (rng.random((rows, S)) * np.exp2(rng.integers(-40, 40, size=(rows, S)))).astype(np.float32)
    scales[0, 0], scales[0, 1], scales[1, 0], scales[1, 1] = 1.0, 0.0, 2.0 ** -20, 2.0 ** 20
    got = orc.ll_dequant(codes, scales)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32)
    sc = torch.from_numpy(scales).repeat_interleave(128, dim=1)
    exp = _bits((dec * sc).to(torch.bfloat16))
    nan = torch.isnan(dec).numpy()
    np.testing.assert_array_equal(got[~nan], exp[~nan])
    # the two NaN codes (0x7F, 0xFF) decode to NaN
    assert np.isnan(torch.from_numpy(got[nan].view(np.int16)).view(torch.bfloat16).float().numpy()).all()
    # every code was exercised in blocks with different scales
    assert len(np.unique(codes)) == 256


def test_ll_dequant_of_the_quantiser_bound(orc):
    """Dequantised codes of real rows stay within 2^-4 |x| + 2^-10 scale of x
    (e4m3 keeps 3 mantissa bits; subnormal step 2^-9 of the scale)."""
    rng = np.random.default_rng(4)
    x = (torch.from_numpy(rng.standard_normal((6, 256)) * np.exp2(rng.integers(-8, 8, size=(6, 1))))
         .to(torch.bfloat16))
    xb = _bits(x)
    for r in range(6):
        codes, scales = orc.quantize_row(xb[r])
        y = orc.ll_dequant(codes[None], scales[None])[0]
        yv = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).double().numpy()
        xv = x[r].double().numpy()
        bound = 2.0 ** -4 * np.abs(xv) + 2.0 ** -10 * np.repeat(scales.astype(np.float64), 128) \
            + 2.0 ** -8 * np.abs(yv)  # the final bf16 rounding
        assert (np.abs(yv - xv) <= bound).all()


# ---------------------------------------------------------------------------
# hierarchical staging
# ---------------------------------------------------------------------------

HIER_CASES = [
    # (R, N, E, K, T, H, mask_p, distinct, seed)
    (4, 2, 8, 2, 6, 16, 0.0, True, 0),
    (8, 2, 16, 3, 9, 8, 0.2, True, 1),
    (8, 4, 32, 4, 7, 8, 0.1, False, 2),    # duplicates
    (6, 3, 12, 2, 5, 8, 0.3, True, 3),
]


def _hier(orc, R, N, E, K, T, H, mask_p, distinct, seed):
    idx = inputs.random_topk(R, E, K, T, seed, mask_p, distinct)
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    lay = orc.layout(idx, R, E, num_nodes=N)
    note = orc.notify(lay, R, E, T, 2)
    sb, sp = orc.hier_stage_pos(lay, R, T, N)
    st = orc.hier_dispatch(x, lay, note, sb, sp, R, N)
    flat = orc.dispatch(x, idx, w, note, R, E)
    return idx.numpy(), _bits(x), lay, note, sb, sp, st, flat


@pytest.mark.parametrize("case", HIER_CASES, ids=[f"h{c[-1]}" for c in HIER_CASES])
def test_hier_stage_a_rows_against_enumeration(orc, case):
    R, N, E, K, T, H, mask_p, distinct, seed = case
    idx, xb, lay, note, sb, sp, st, flat = _hier(orc, *case)
    ref, _ = pyref.layout(idx, R, E, N)
    pos, base = pyref.stage_positions(ref["is_token_in_node"], R, N)
    np.testing.assert_array_equal(sb, base)
    assert st["staging"].shape[0] == len(pos)
    for (s, t, n), p in pos.items():
        assert sp[s, t, n] == p
        np.testing.assert_array_equal(st["staging"][p], xb[s, t], err_msg=f"staged row of ({s}, {t}, node {n})")
        assert st["stage_src_rank"][p] == s and st["stage_src_idx"][p] == t


@pytest.mark.parametrize("case", HIER_CASES, ids=[f"h{c[-1]}" for c in HIER_CASES])
def test_hier_stage_b_rows_against_receive_lists(orc, case):
    R, N, E, K, T, H, mask_p, distinct, seed = case
    idx, xb, lay, note, sb, sp, st, flat = _hier(orc, *case)
    ref, _ = pyref.layout(idx, R, E, N)
    _, lists = pyref.send_pos(ref["is_token_in_rank"])
    base = 0
    for d in range(R):
        for i, (s, t) in enumerate(lists[d]):
            np.testing.assert_array_equal(st["recv_x"][base + i], xb[s, t], err_msg=f"rank {d} row {i}")
        base += len(lists[d])
    assert st["recv_x"].shape[0] == base
    # and the staged path lands exactly where the flat dispatch does
    np.testing.assert_array_equal(st["recv_x"], flat["recv_x"])


def test_hier_worked_case_staged_equals_flat(orc):
    G = load("worked_r4e8.txt")
    R, E, K, T, C, N = (int(G[k]) for k in ("R", "E", "K", "T", "C", "N"))
    idx = np.full((R, T, K), -1, np.int64)
    idx[0] = G["topk_idx[0]"].astype(np.int64)
    x = inputs.random_x(R, T, 128, 21)
    w = inputs.random_weights(R, T, K, 21)
    xb = _bits(x)
    lay = orc.layout(idx, R, E, num_nodes=N)
    note = orc.notify(lay, R, E, T, C)
    sb, sp = orc.hier_stage_pos(lay, R, T, N)
    st = orc.hier_dispatch(x, lay, note, sb, sp, R, N)
    # staged rows: stage_pos[0] = t0:(0,-1) t1:(1,3) t2:(-1,4) t3:(2,5)
    for t, p in ((0, 0), (1, 1), (3, 2), (1, 3), (2, 4), (3, 5)):
        np.testing.assert_array_equal(st["staging"][p], xb[0, t])
    # forwarded rows, in the worked receive order recv_src_idx = 0 1 3 1 2 3
    for r, t in enumerate(G["recv_src_idx"].astype(int)):
        np.testing.assert_array_equal(st["recv_x"][r], xb[0, t])
    np.testing.assert_array_equal(st["recv_x"], orc.dispatch(x, idx, w, note, R, E)["recv_x"])
