"""Invariants the definitions fix, checked on the oracle over random and edge-case routings.

* sum over experts of num_tokens_per_expert equals the number of valid entries;
* num_tokens_per_rank is the row sum of is_token_in_rank, and never exceeds the
  valid entries (equality iff no token has two experts on one rank);
* channel_prefix_matrix ends at num_tokens_per_rank and never decreases;
* the ragged offsets are exclusive prefix sums of the received counts;
* send positions are a bijection onto each receiver's block; permuted rows are
  a bijection with the valid pairs;
* combine(permute(dispatch(x))) with the identity expert and weights summing to
  one gives x back; with masked entries it gives x * (sum of valid weights);
* low-latency slot addresses never collide and every count slot is written.
"""
import numpy as np
import pytest
import torch

import pyref

from combine_get_dispatch_histograms_gb300 import inputs

CASES = [
    # (R, E, K, T, H, C, mask_p, distinct, seed)
    (4, 8, 2, 16, 128, 2, 0.0, True, 0),
    (4, 8, 2, 37, 64, 3, 0.2, True, 1),      # ragged channels, masks
    (8, 64, 8, 50, 32, 8, 0.05, True, 2),
    (2, 4, 4, 9, 16, 4, 0.0, False, 3),      # duplicate experts inside a token
    (3, 9, 3, 0, 16, 2, 0.0, True, 4),       # no tokens at all
    (4, 16, 4, 5, 16, 8, 1.0, True, 5),      # every entry masked; more channels than tokens
    (1, 4, 2, 7, 16, 2, 0.1, True, 6),       # a single rank
]


def _run(orc, R, E, K, T, H, C, mask_p, distinct, seed):
    idx = inputs.random_topk(R, E, K, T, seed, mask_p, distinct)
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    lay = orc.layout(idx, R, E)
    note = orc.notify(lay, R, E, T, C)
    disp = orc.dispatch(x, idx, w, note, R, E)
    perm = orc.permute(idx, disp["recv_x"], note, R, E)
    return idx.numpy(), x, w, lay, note, disp, perm


@pytest.mark.parametrize("case", CASES)
def test_layout_and_notify_invariants(orc, case):
    R, E, K, T, H, C, mask_p, distinct, seed = case
    idx, x, w, lay, note, disp, perm = _run(orc, *case)
    L = E // R
    valid = idx >= 0
    ntpe, ntpr, itir = lay["num_tokens_per_expert"], lay["num_tokens_per_rank"], lay["is_token_in_rank"]
    np.testing.assert_array_equal(ntpe.sum(axis=1), valid.reshape(R, -1).sum(axis=1))
    np.testing.assert_array_equal(ntpr, itir.sum(axis=1))
    per_src_valid = valid.reshape(R, -1).sum(axis=1)
    assert (ntpr.sum(axis=1) <= per_src_valid).all()
    ranks = np.where(valid, idx // L, -1)
    for s in range(R):
        two_on_one = any(len(set(r[r >= 0].tolist())) < (r >= 0).sum() for r in ranks[s])
        assert (ntpr[s].sum() == per_src_valid[s]) == (not two_on_one)
    cpm = note["channel_prefix_matrix"]
    np.testing.assert_array_equal(cpm[:, :, -1], ntpr)
    assert (np.diff(cpm, axis=2) >= 0).all()
    rc, ro = note["recv_count"], note["recv_offsets"]
    np.testing.assert_array_equal(rc, ntpr.T)
    np.testing.assert_array_equal(ro[:, 0], 0)
    np.testing.assert_array_equal(ro[:, 1:], np.cumsum(rc, axis=1)[:, :-1])
    np.testing.assert_array_equal(ro[:, -1] + rc[:, -1], note["num_recv_tokens"])
    np.testing.assert_array_equal(note["rank_base"], np.concatenate([[0], np.cumsum(note["num_recv_tokens"])]))
    np.testing.assert_array_equal(note["num_recv_per_expert"], ntpe.sum(axis=0).reshape(R, L))
    sp = note["send_pos"]
    for d in range(R):
        got = np.sort(sp[:, :, d][sp[:, :, d] >= 0])
        np.testing.assert_array_equal(got, np.arange(note["num_recv_tokens"][d]))
    P = int(valid.sum())
    assert note["perm_rank_base"][R] == P
    pp = perm["perm_pos"]
    assert ((pp >= 0) == valid).all()
    np.testing.assert_array_equal(np.sort(pp[pp >= 0]), np.arange(P))
    # every permuted row is a copy of its source token
    xb = x.view(torch.int16).numpy().view(np.uint16)
    for s, t, k in zip(*np.nonzero(valid)):
        np.testing.assert_array_equal(perm["permuted_x"][pp[s, t, k]], xb[s, t])
        np.testing.assert_array_equal(disp["recv_x"][perm["perm_src_row"][pp[s, t, k]]], xb[s, t])


@pytest.mark.parametrize("case", CASES)
def test_combine_identity_expert(orc, case):
    R, E, K, T, H, C, mask_p, distinct, seed = case
    idx, x, w, lay, note, disp, perm = _run(orc, *case)
    valid = idx >= 0
    # weights renormalised over the valid entries sum to one (up to fp32 rounding)
    wn = np.where(valid, w.numpy(), 0).astype(np.float64)
    sums = wn.sum(axis=2, keepdims=True)
    wn = np.where(sums > 0, wn / np.where(sums > 0, sums, 1), 0).astype(np.float32)
    wn = np.where(valid, wn, w.numpy())  # masked weights stay as drawn but are unused
    out = orc.combine(perm["permuted_x"], perm["perm_pos"], idx, wn, R, E, "ord32")
    xb = x.view(torch.int16).numpy().view(np.uint16)
    has = valid.any(axis=2)
    # tokens with a valid entry come back bit-exactly; bf16 values are far from
    # bf16 midpoints, so x * (1 +- a few fp32 ulps) rounds back to x (-0 -> +0)
    expect = np.where(xb == 0x8000, 0, xb)
    np.testing.assert_array_equal(out[has], expect[has])
    assert (out[~has] == 0).all()  # tokens sent nowhere combine to +0


@pytest.mark.parametrize("case", CASES[:4])
def test_combine_masked_closed_form_and_ref64(orc, case):
    R, E, K, T, H, C, mask_p, distinct, seed = case
    idx, x, w, lay, note, disp, perm = _run(orc, *case)
    valid = idx >= 0
    o32 = orc.combine(perm["permuted_x"], perm["perm_pos"], idx, w, R, E, "ord32")
    o64 = orc.combine(perm["permuted_x"], perm["perm_pos"], idx, w, R, E, "ref64")
    f32 = torch.from_numpy(o32.view(np.int16)).view(torch.bfloat16).float().numpy()
    f64 = torch.from_numpy(o64.view(np.int16)).view(torch.bfloat16).float().numpy()
    closed = x.float().numpy().astype(np.float64) * np.where(valid, w.numpy(), 0).sum(axis=2, keepdims=True)
    tol = 1e-2 + 4e-3 * np.abs(closed)
    assert (np.abs(f32 - closed) <= tol + np.abs(closed) * 2.0 ** -8).all()
    # ord32 and ref64 differ at most by one bf16 ulp (a rounding-midpoint flip)
    ulp = np.maximum(np.abs(f64), 2.0 ** -126) * 2.0 ** -7
    assert (np.abs(f32 - f64) <= ulp).all()


def test_low_latency_invariants(orc):
    R, E, K, T, H, cap = 4, 16, 4, 24, 256, 24
    idx = inputs.random_topk(R, E, K, T, 9, 0.1)
    x = inputs.random_x(R, T, H, 9)
    sent = orc.ll_send(x, idx, R, E, cap)
    valid = idx.numpy() >= 0
    assert (sent["counts"] >= 0).all()
    assert sent["counts"].sum() == valid.sum()
    s_, t_, k_ = np.nonzero(valid)
    e_ = idx.numpy()[s_, t_, k_]
    addr = (e_ * R + s_) * cap + sent["slot"][s_, t_, k_]
    assert len(np.unique(addr)) == len(addr) and addr.max() < E * R * cap
    pk = orc.ll_pack(sent, R, E, H, cap)
    L = E // R
    np.testing.assert_array_equal(pk["packed_recv_count"].reshape(-1), sent["counts"].sum(axis=1))
    lr = pk["layout_range"]
    np.testing.assert_array_equal(lr[..., 1], sent["counts"].reshape(R, L, R))
    np.testing.assert_array_equal(lr[..., 0], np.cumsum(lr[..., 1], axis=2) - lr[..., 1])
    # packed rows carry the codes of their source token
    xb = x.view(torch.int16).numpy().view(np.uint16)
    for s, t, k in list(zip(s_, t_, k_))[:50]:
        e = idx[s, t, k].item()
        d, l = divmod(e, L)
        row = lr[d, l, s, 0] + sent["slot"][s, t, k]
        codes, scales = orc.quantize_row(xb[s, t])
        np.testing.assert_array_equal(pk["packed_x"][d, l, row], codes)
        np.testing.assert_array_equal(pk["packed_scales"][d, l, row], scales)
        assert tuple(pk["packed_src_info"][d, l, row]) == (s, t)


def test_low_latency_microbatches_closed_form(orc):
    """Splitting T into microbatches of <= cap tokens only changes the slots'
    origin; each microbatch combines its own rows.  With the identity expert
    every entry of a token carries the same dequantised row, so the result
    has a closed form: for k ascending over the valid entries,
    acc = fma(w[s][t][k], y[s][t], acc) in fp32, then bf16, where y[s][t] is
    the token's quantised row decoded by torch.float8_e4m3fn times its
    block's scale (fp32) and rounded to bf16."""
    R, E, K, T, H = 2, 8, 2, 10, 128
    idx = inputs.random_topk(R, E, K, T, 11, 0.1)
    x = inputs.random_x(R, T, H, 11)
    w = inputs.random_weights(R, T, K, 11)
    out = np.zeros((R, T, H), np.uint16)
    for t0, n in ((0, 4), (4, 4), (8, 2)):
        sent = orc.ll_send(x, idx, R, E, 4, t0, n)
        assert sent["counts"].sum() == (idx.numpy()[:, t0:t0 + n] >= 0).sum()
        pk = orc.ll_pack(sent, R, E, H, 4)
        y = orc.ll_dequant(pk["packed_x"], pk["packed_scales"])
        orc.ll_combine(y, idx, w, sent["slot"], pk["layout_range"], R, E, 4, t0, n, out=out)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    idn, wn = idx.numpy(), w.numpy()
    for s in range(R):
        for t in range(T):
            codes, scales = orc.quantize_row(xb[s, t])
            dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).float()
            yq = (dec * torch.from_numpy(scales).repeat_interleave(128)).to(torch.bfloat16).float().tolist()
            ks = [k for k in range(K) if idn[s, t, k] >= 0]
            for j in range(H):
                acc = 0.0
                for k in ks:
                    acc = pyref.fmaf(float(wn[s, t, k]), yq[j], acc)
                assert out[s, t, j] == pyref.bf16_bits_of(acc), (s, t, j)


def test_size_hint(orc):
    for cap, H, R, E in ((128, 7168, 16, 256), (256, 4096, 32, 256), (6, 128, 4, 8)):
        hint = orc.ll_size_hint(cap, H, R, E)
        msg = orc.ll_message_bytes(H)
        assert msg >= 16 + H + H // 128 * 4 and msg % 16 == 0
        need = 2 * (E * R * cap * msg + E * R * 4)
        assert hint >= need and hint % 128 == 0 and hint - need < 2 * (128 + 16)


def test_invalid_topk_reported(orc):
    idx = np.zeros((2, 3, 2), np.int64)
    idx[1, 2, 0] = 9
    with pytest.raises(orc.OracleError) as e:
        orc.layout(idx, 2, 4)
    assert e.value.code == -2


@pytest.mark.parametrize("case", CASES, ids=[f"c{c[-1]}" for c in CASES])
@pytest.mark.parametrize("align", [1, 3, 16, 128])
def test_expert_alignment(orc, case, align):
    """Expert-aligned permuted layout: every (rank, local expert) block starts at
    a multiple of the alignment inside its rank and takes its count rounded up;
    dropping the padding rows gives the unaligned layout row for row; padding
    rows are marked -1 and referenced by no pair; everything else in the
    handle is as without alignment."""
    R, E, K, T, H, C, mask_p, distinct, seed = case
    idx, x, w, lay, note1, disp, perm1 = _run(orc, *case)
    L = E // R
    note = orc.notify(lay, R, E, T, C, align=align)
    for k in ("recv_count", "num_recv_tokens", "recv_offsets", "rank_base", "num_recv_per_expert",
              "channel_prefix_matrix", "send_pos"):
        assert np.array_equal(note[k], note1[k]), k
    cnt = note["num_recv_per_expert"].astype(np.int64)
    padded = (cnt + align - 1) // align * align
    eo = note["expert_offsets"].astype(np.int64)
    assert (eo % align == 0).all()
    assert (eo[:, 0] == 0).all()
    assert np.array_equal(eo[:, 1:] - eo[:, :-1], padded[:, :-1])
    prb = note["perm_rank_base"].astype(np.int64)
    assert prb[0] == 0 and np.array_equal(np.diff(prb), padded.sum(axis=1))
    if align == 1:
        assert np.array_equal(eo, note1["expert_offsets"]) and np.array_equal(prb, note1["perm_rank_base"])
    perm = orc.permute(idx, disp["recv_x"], note, R, E)
    pp = perm["perm_pos"]
    psr = perm["perm_src_row"]
    P = int(prb[R])
    assert psr.shape == (P,)
    # every pair lands inside its own block, in (s, t, k) order
    used = np.zeros(P, bool)
    last = {}
    for s, t, k in zip(*np.nonzero(idx >= 0)):
        e = int(idx[s, t, k])
        d, l = divmod(e, L)
        r = int(pp[s, t, k])
        lo = prb[d] + eo[d, l]
        assert lo <= r < lo + cnt[d, l], (s, t, k)
        assert not used[r]
        used[r] = True
        assert last.get((d, l), -1) < r
        last[(d, l)] = r
    assert np.array_equal(psr >= 0, used)
    # without the padding rows: the unaligned layout, row for row
    assert np.array_equal(psr[used], perm1["perm_src_row"])
    assert np.array_equal(perm["permuted_x"][used], perm1["permuted_x"])
    # the unaligned perm_pos is the aligned one renumbered over the used rows
    rank_of = np.cumsum(used) - 1
    valid = idx >= 0
    assert np.array_equal(rank_of[pp[valid]], perm1["perm_pos"][valid])
