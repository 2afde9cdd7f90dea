"""Parity at the full workload sizes, in the launch configuration bench.py
times (same Context / LLBuffer parameters).

The oracle computes every integer result exactly at full size (layout, notify,
handle, positions, slots, counts; its copy steps run on an 8-channel stand-in
of x, since positions do not depend on H).  Row data is checked for every row
against the row the oracle assigned (a GPU gather of x does the data movement
of the comparison); combine outputs are checked bit-exactly on sampled tokens,
each computed by the oracle on a sub-problem holding only those tokens with
the same experts, weights and summation order."""
import numpy as np
import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, LLBuffer, inputs
from parity_util import eq, bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_SAMPLES = 384


def _rows_equal(got: torch.Tensor, src: torch.Tensor, src_rows: np.ndarray, what: str, chunk=1 << 15):
    """got[i] == src[src_rows[i]] for every i (compared on the GPU, in chunks)."""
    assert got.shape[0] == len(src_rows), what
    idx = torch.from_numpy(src_rows.astype(np.int64)).to(got.device)
    for a in range(0, len(src_rows), chunk):
        b = min(len(src_rows), a + chunk)
        exp = src.index_select(0, idx[a:b])
        if not torch.equal(got[a:b].view(torch.int16), exp.view(torch.int16)):
            bad = (got[a:b].view(torch.int16) != exp.view(torch.int16)).any(dim=1).nonzero()
            raise AssertionError(f"{what}: row {a + int(bad[0])} differs ({len(bad)} rows in chunk)")


def _normal_full(wl, hier: bool):
    R, E, K, T, H, C, N = wl.R, wl.E, wl.K, wl.T, wl.H, wl.num_channels, wl.num_nodes
    idx, w = inputs.make_routing(wl, 0)
    x = inputs.make_x(wl, 0, device="cuda")
    xf = x.view(R * T, H)
    ctx = Context(R, E, K, T, H, num_channels=C, num_nodes=N)
    idxd, wd = idx.cuda(), w.cuda()
    lay = ctx.get_dispatch_layout(idxd, nodes=N > 1)
    h = ctx.notify_dispatch(idxd, lay)
    recv = ctx.dispatch_hier(x, idxd, wd, h) if hier else ctx.dispatch(x, idxd, wd, h)
    perm = ctx.permute(h, recv)
    out = ctx.combine(h, perm["permuted_x"], idxd, wd, hier=hier)
    ctx.check()
    torch.cuda.synchronize()

    # ---- integers, exactly, at full size ------------------------------------------
    o_lay = orc.layout(idx, R, E, num_nodes=N if N > 1 else 0)
    for k in o_lay:
        eq(lay[k], o_lay[k], k)
    o_note = orc.notify(o_lay, R, E, T, C)
    for k in ("recv_count", "num_recv_tokens", "recv_offsets", "rank_base", "num_recv_per_expert",
              "expert_offsets", "perm_rank_base", "channel_prefix_matrix", "send_pos"):
        eq(h[k], o_note[k], k)
    # the oracle's copy steps on an 8-channel stand-in give the metadata exactly
    probe = np.zeros((R, T, 8), np.uint16)
    o_disp = orc.dispatch(probe, idx, w, o_note, R, E)
    for k in ("recv_src_rank", "recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        eq(recv[k], o_disp[k], k)
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    eq(h["perm_pos"], o_perm["perm_pos"], "perm_pos")
    eq(perm["perm_src_row"], o_perm["perm_src_row"], "perm_src_row")

    # ---- every row of data ---------------------------------------------------------
    src_tok = o_disp["recv_src_rank"].astype(np.int64) * T + o_disp["recv_src_idx"]
    _rows_equal(recv["recv_x"], xf, src_tok, "recv_x")
    _rows_equal(perm["permuted_x"], xf, src_tok[o_perm["perm_src_row"]], "permuted_x")
    if not hier:
        del recv
        fused = ctx.dispatch_permuted(x, idxd, wd, h)
        ctx.check()
        eq(fused["perm_src_token"], src_tok[o_perm["perm_src_row"]].astype(np.int32), "perm_src_token")
        _rows_equal(fused["permuted_x"], xf, src_tok[o_perm["perm_src_row"]], "permuted_x (fused dispatch)")
        del fused
    if hier:
        sb, sp = orc.hier_stage_pos(o_lay, R, T, N)
        eq(h["stage_base"], sb, "stage_base")
        eq(h["stage_pos"], sp, "stage_pos")
        o_st = orc.hier_dispatch(probe, o_lay, o_note, sb, sp, R, N)
        eq(recv["stage_src_rank"], o_st["stage_src_rank"], "stage_src_rank")
        eq(recv["stage_src_idx"], o_st["stage_src_idx"], "stage_src_idx")
        st_tok = o_st["stage_src_rank"].astype(np.int64) * T + o_st["stage_src_idx"]
        _rows_equal(recv["staging"], xf, st_tok, "staging")

    # ---- combine on sampled tokens ----------------------------------------------
    rng = np.random.default_rng(7)
    g = rng.choice(R * T, size=min(N_SAMPLES, R * T), replace=False)
    m = len(g)
    idx_np, w_np = idx.numpy().reshape(R * T, K), w.numpy().reshape(R * T, K)
    sub_idx = np.full((R, m, K), -1, np.int64)
    sub_w = np.zeros((R, m, K), np.float32)
    sub_idx[0], sub_w[0] = idx_np[g], w_np[g]
    sub_pp = np.full((R, m, K), -1, np.int32)
    sub_pp[0] = (np.arange(m)[:, None] * K + np.arange(K)[None, :]).astype(np.int32)
    xs = bits(xf.index_select(0, torch.from_numpy(g).cuda()))          # identity expert: rows are x
    y_sub = np.repeat(xs, K, axis=0)
    if hier:
        exp = orc.combine_hier(y_sub, sub_pp, sub_idx, sub_w, R, E, N)[0]
    else:
        exp = orc.combine(y_sub, sub_pp, sub_idx, sub_w, R, E, "ord32")[0]
    got = bits(out.view(R * T, H).index_select(0, torch.from_numpy(g).cuda()))
    eq(got, exp, "combine (sampled tokens)")
    return ctx


def test_prefill_full():
    _normal_full(inputs.WORKLOADS["prefill"], hier=False)


def test_skewed_normal_full():
    _normal_full(inputs.WORKLOADS["skewed"], hier=False)


def test_hier_full_staged():
    _normal_full(inputs.WORKLOADS["hier"], hier=True)


def _ll_full(wl):
    R, E, K, T, H, cap = wl.R, wl.E, wl.K, wl.T, wl.H, wl.ll_cap
    L = E // R
    idx, w = inputs.make_routing(wl, 0)
    x = inputs.make_x(wl, 0, device="cuda")
    xf = x.view(R * T, H)
    buf = LLBuffer(R, E, K, T, H, cap)
    idxd, wd = idx.cuda(), w.cuda()
    out = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
    pk = buf.alloc_packed()
    y_ll = torch.empty(pk["packed_x"].shape, dtype=torch.bfloat16, device="cuda")
    probe = np.zeros((R, T, 128), np.uint16)
    rng = np.random.default_rng(11)
    for t0 in range(0, T, cap):
        n = min(cap, T - t0)
        buf.dispatch(x, idxd, t0, n, out=pk)
        buf.check()
        # identity expert (the expert is not part of the path): y = bf16(code * scale)
        for d in range(R):
            y_ll[d] = (pk["packed_x"][d].view(torch.float8_e4m3fn).float() *
                       pk["packed_scales"][d].repeat_interleave(128, dim=-1)).to(torch.bfloat16)
        buf.combine(y_ll, idxd, wd, pk, t0, n, out=out)
        buf.check()
        # integers exactly (slots do not depend on H: the oracle runs on a 128-channel stand-in)
        sent = orc.ll_send(probe, idx, R, E, cap, t0, n)
        o_pk = orc.ll_pack(sent, R, E, 128, cap)
        eq(pk["slot"][:, t0:t0 + n], sent["slot"][:, t0:t0 + n], "slot")
        eq(pk["packed_recv_count"], o_pk["packed_recv_count"], "packed_recv_count")
        eq(pk["layout_range"], o_pk["layout_range"], "layout_range")
        # sampled messages: codes, scales and source of valid (s, t, k)
        s_, t_, k_ = np.nonzero(idx.numpy()[:, t0:t0 + n] >= 0)
        pick = rng.choice(len(s_), size=min(N_SAMPLES, len(s_)), replace=False)
        lr = o_pk["layout_range"]
        for j in pick[:64]:
            s, t, k = int(s_[j]), int(t0 + t_[j]), int(k_[j])
            e = int(idx[s, t, k])
            d, l = divmod(e, L)
            row = lr[d, l, s, 0] + sent["slot"][s, t, k]
            codes, scales = orc.quantize_row(bits(xf[s * T + t]))
            eq(pk["packed_x"][d, l, row], codes, f"packed_x ({s},{t},{k})")
            eq(pk["packed_scales"][d, l, row], scales, f"packed_scales ({s},{t},{k})")
            assert tuple(pk["packed_src_info"][d, l, row].tolist()) == (s, t)
        # sampled tokens of the microbatch: the oracle's k-ordered fp32 sum on a
        # one-rank sub-problem (one expert per k, one slot per token)
        toks = rng.choice(R * n, size=min(128, R * n), replace=False)
        gs = [(int(q // n), int(t0 + q % n)) for q in toks]
        m = len(gs)
        sub_idx = np.full((1, m, K), -1, np.int64)
        sub_w = np.zeros((1, m, K), np.float32)
        sub_slot = np.full((1, m, K), -1, np.int32)
        y_sub = np.zeros((1, K, m, H), np.uint16)
        for i, (s, t) in enumerate(gs):
            codes, scales = orc.quantize_row(bits(xf[s * T + t]))
            yrow = orc.ll_dequant(codes[None], scales[None])[0]
            for k in range(K):
                if idx[s, t, k] >= 0:
                    sub_idx[0, i, k] = k
                    sub_w[0, i, k] = w[s, t, k]
                    sub_slot[0, i, k] = i
                    y_sub[0, k, i] = yrow
        sub_lr = np.zeros((1, K, 1, 2), np.int32)
        sub_lr[..., 1] = m
        exp = orc.ll_combine(y_sub, sub_idx, sub_w, sub_slot, sub_lr, 1, K, m)[0]
        got = np.stack([bits(out[s, t]) for s, t in gs])
        eq(got, exp, f"ll combine (sampled tokens, microbatch {t0})")


def test_decode_ll_full():
    _ll_full(inputs.WORKLOADS["decode"])


def test_skewed_ll_full_microbatches():
    _ll_full(inputs.WORKLOADS["skewed"])


def test_prefill_full_fp8_one_pass():
    """The one-pass FP8 dispatches at the prefill size, in the bench's launch
    configuration: every pair row equals the two-pass form (quantise, then the
    fused FP8 dispatch) byte for byte, and sampled rows equal the oracle's
    quantisation of their source token."""
    wl = inputs.WORKLOADS["prefill"]
    R, E, K, T, H, C = wl.R, wl.E, wl.K, wl.T, wl.H, wl.num_channels
    idx, w = inputs.make_routing(wl, 0)
    x = inputs.make_x(wl, 0, device="cuda")
    ctx = Context(R, E, K, T, H, num_channels=C)
    idxd, wd = idx.cuda(), w.cuda()
    h = ctx.notify_dispatch(idxd, ctx.get_dispatch_layout(idxd))
    n_def = H + H // 32
    one = ctx.dispatch_permuted_quant(x, idxd, wd, h)
    xq = ctx.quantize_fp8(x)
    two = ctx.dispatch_permuted_fp8(xq, idxd, wd, h)
    ctx.check()
    assert torch.equal(one["permuted_xq"][:, :n_def], two["permuted_xq"][:, :n_def])
    assert torch.equal(one["perm_src_token"], two["perm_src_token"])
    assert torch.equal(one["perm_weight"], two["perm_weight"])
    recv = ctx.dispatch_quant(x, idxd, wd, h)
    recv2 = ctx.dispatch_fp8(xq, idxd, wd, h)
    ctx.check()
    assert torch.equal(recv["recv_xq"][:, :n_def], recv2["recv_xq"][:, :n_def])
    for k in ("recv_src_rank", "recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        assert torch.equal(recv[k], recv2[k]), k
    # sampled rows against the oracle's quantisation of their source token
    rng = np.random.default_rng(3)
    rows = rng.choice(one["permuted_xq"].shape[0], size=256, replace=False)
    src = one["perm_src_token"].cpu().numpy()[rows]
    xf = x.view(R * T, H)
    got = bits(one["permuted_xq"][torch.from_numpy(rows).cuda()])
    for i, g in enumerate(src):
        codes, scales = orc.quantize_row(bits(xf[int(g)]))
        eq(got[i, :H], codes, f"codes of row {rows[i]}")
        eq(got[i, H:n_def].view(np.float32), scales, f"scales of row {rows[i]}")
