"""Parity at the full workload sizes, in the launch configuration bench.py
times (same Context / LLBuffer parameters).

The oracle computes every integer result exactly at full size (layout, notify,
handle, positions, slots, counts; its copy steps run on an 8-channel stand-in
of x, since positions do not depend on H).  Row data is checked for every row
against the row the oracle assigned (a GPU gather of x does the data movement
of the comparison); every FP8 row and message is checked against the oracle's
quantisation of its source token.  Combine outputs are checked bit-exactly on
sampled tokens, each computed by the oracle on a sub-problem holding only
those tokens with the same experts, weights and summation order, for the
identity expert and for an expert output with a distinct row per permuted
row or packed slot."""
import numpy as np
import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, LLBuffer, inputs
from parity_util import eq, bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_SAMPLES = 384


def _rows_equal(got: torch.Tensor, src: torch.Tensor, src_rows: np.ndarray, what: str, chunk=1 << 15,
                got_rows: np.ndarray = None):
    """got[i] == src[src_rows[i]] for every i, or got[got_rows[i]] ==
    src[src_rows[i]] when got_rows is given (compared byte for byte on the
    GPU, in chunks)."""
    if got_rows is None:
        assert got.shape[0] == len(src_rows), what
    else:
        assert len(got_rows) == len(src_rows), what
        gidx = torch.from_numpy(got_rows.astype(np.int64)).to(got.device)
    idx = torch.from_numpy(src_rows.astype(np.int64)).to(got.device)
    for a in range(0, len(src_rows), chunk):
        b = min(len(src_rows), a + chunk)
        exp = src.index_select(0, idx[a:b]).contiguous().view(torch.uint8)
        g = (got[a:b] if got_rows is None else got.index_select(0, gidx[a:b])).contiguous().view(torch.uint8)
        if not torch.equal(g, exp):
            bad = (g != exp).any(dim=1).nonzero()
            raise AssertionError(f"{what}: row {a + int(bad[0])} differs ({len(bad)} rows in chunk)")


def _oracle_fp8_rows(xf: torch.Tensor) -> torch.Tensor:
    """The oracle's FP8 row (H codes, then H/128 fp32 scales as bytes) of
    every token of xf [N][H], on the GPU for the gathers."""
    codes, scales = orc.quantize_rows(bits(xf))
    return torch.from_numpy(np.concatenate([codes, scales.view(np.uint8)], axis=1)).to(xf.device)


def _combine_sub_problem(y_rows: np.ndarray, idx_np, w_np, g, R, E, K, hier, N):
    """The oracle's combine of the sampled tokens g: one sub-problem holding
    only those tokens (on source 0) with their experts, weights and the rows
    y_rows [m][K][H] their entries read (rows of masked entries unused)."""
    m = len(g)
    H = y_rows.shape[2]
    sub_idx = np.full((R, m, K), -1, np.int64)
    sub_w = np.zeros((R, m, K), np.float32)
    sub_idx[0], sub_w[0] = idx_np[g], w_np[g]
    sub_pp = np.full((R, m, K), -1, np.int32)
    sub_pp[0] = (np.arange(m)[:, None] * K + np.arange(K)[None, :]).astype(np.int32)
    y_sub = y_rows.reshape(m * K, H)
    if hier:
        return orc.combine_hier(y_sub, sub_pp, sub_idx, sub_w, R, E, N)[0]
    return orc.combine(y_sub, sub_pp, sub_idx, sub_w, R, E, "ord32")[0]


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
    gd = torch.from_numpy(g).cuda()
    idx_np, w_np = idx.numpy().reshape(R * T, K), w.numpy().reshape(R * T, K)
    xs = bits(xf.index_select(0, gd))          # identity expert: every entry's row is x
    exp = _combine_sub_problem(np.repeat(xs[:, None, :], K, axis=1), idx_np, w_np, g, R, E, K, hier, N)
    got = bits(out.view(R * T, H).index_select(0, gd))
    eq(got, exp, "combine (sampled tokens)")
    # an expert output with a distinct row per permuted row: each entry of a
    # sampled token reads its own row, located by the oracle's perm_pos
    P = int(o_note["perm_rank_base"][R])
    del perm, out
    y = inputs.random_rows(P, H, seed=99, device="cuda")
    out_y = ctx.combine(h, y, idxd, wd, hier=hier)
    ctx.check()
    pp = o_perm["perm_pos"].reshape(R * T, K)[g]
    rows = bits(y.index_select(0, torch.from_numpy(np.maximum(pp, 0).reshape(-1)).cuda().long()))
    exp = _combine_sub_problem(rows.reshape(m, K, H), idx_np, w_np, g, R, E, K, hier, N)
    got = bits(out_y.view(R * T, H).index_select(0, gd))
    eq(got, exp, "combine of distinct expert rows (sampled tokens)")
    return ctx


def test_prefill_full():
    _normal_full(inputs.WORKLOADS["prefill"], hier=False)


def test_skewed_normal_full():
    _normal_full(inputs.WORKLOADS["skewed"], hier=False)


def test_hier_full_staged():
    _normal_full(inputs.WORKLOADS["hier"], hier=True)


def _identity_y(pk, R):
    """The identity expert on the packed messages: y = bf16(code * scale)."""
    y = torch.empty(pk["packed_x"].shape, dtype=torch.bfloat16, device="cuda")
    for d in range(R):
        y[d] = (pk["packed_x"][d].view(torch.float8_e4m3fn).float() *
                pk["packed_scales"][d].repeat_interleave(128, dim=-1)).to(torch.bfloat16)
    return y


def _check_ll_microbatch_full(pk, outs, xf, q, idx, w, R, E, K, T, H, cap, t0, n, rng, what=""):
    """Every message of the microbatch against the oracle's quantisation of its
    source token (codes, scales, source), the slots and the receive layout
    exactly, and sampled tokens of each combine output against the oracle's
    k-ordered sum.  outs: [(out, y, y_is_identity)]."""
    L = E // R
    idx_np, w_np = idx.numpy(), w.numpy()
    # integers exactly (slots do not depend on H: the oracle runs on a 128-channel stand-in)
    sent = orc.ll_send(np.zeros((R, T, 128), np.uint16), idx, R, E, cap, t0, n)
    o_pk = orc.ll_pack(sent, R, E, 128, cap)
    eq(pk["slot"][:, t0:t0 + n], sent["slot"][:, t0:t0 + n], "slot" + what)
    eq(pk["packed_recv_count"], o_pk["packed_recv_count"], "packed_recv_count" + what)
    eq(pk["layout_range"], o_pk["layout_range"], "layout_range" + what)
    # every message of the microbatch: codes, scales and source of each valid (s, t, k)
    s_, t_, k_ = np.nonzero(idx_np[:, t0:t0 + n] >= 0)
    t_ = t_ + t0
    e_ = idx_np[s_, t_, k_]
    d_, l_ = e_ // L, e_ % L
    lr = o_pk["layout_range"]
    row = lr[d_, l_, s_, 0] + sent["slot"][s_, t_, k_]
    msg = (d_ * L + l_) * (R * cap) + row
    tok = s_ * T + t_
    _rows_equal(pk["packed_x"].view(-1, H), q[:, :H], tok, "packed_x (every message)" + what, got_rows=msg)
    _rows_equal(pk["packed_scales"].view(-1, H // 128), q[:, H:].view(torch.float32), tok,
                "packed_scales (every message)" + what, got_rows=msg)
    src_info = torch.from_numpy(np.stack([s_, t_], axis=1).astype(np.int32)).cuda()
    _rows_equal(pk["packed_src_info"].view(-1, 2), src_info, np.arange(len(msg)),
                "packed_src_info (every message)" + what, got_rows=msg)
    # sampled tokens of the microbatch: the oracle's k-ordered fp32 sum on a
    # one-rank sub-problem (one expert per k, one slot per token)
    toks = rng.choice(R * n, size=min(128, R * n), replace=False)
    gs = [(int(qq // n), int(t0 + qq % n)) for qq in toks]
    m = len(gs)
    sub_idx = np.full((1, m, K), -1, np.int64)
    sub_w = np.zeros((1, m, K), np.float32)
    sub_slot = np.full((1, m, K), -1, np.int32)
    sub_lr = np.zeros((1, K, 1, 2), np.int32)
    sub_lr[..., 1] = m
    for out, y, identity in outs:
        y_sub = np.zeros((1, K, m, H), np.uint16)
        yf = y.view(-1, H)
        for i, (s, t) in enumerate(gs):
            if identity:
                codes, scales = orc.quantize_row(bits(xf[s * T + t]))
                yrow = orc.ll_dequant(codes[None], scales[None])[0]
            for k in range(K):
                e = int(idx_np[s, t, k])
                if e >= 0:
                    sub_idx[0, i, k] = k
                    sub_w[0, i, k] = w_np[s, t, k]
                    sub_slot[0, i, k] = i
                    d, l = divmod(e, L)
                    y_sub[0, k, i] = yrow if identity else \
                        bits(yf[(d * L + l) * R * cap + lr[d, l, s, 0] + sent["slot"][s, t, k]])
        exp = orc.ll_combine(y_sub, sub_idx, sub_w, sub_slot, sub_lr, 1, K, m)[0]
        got = np.stack([bits(out[s, t]) for s, t in gs])
        kind = "identity expert" if identity else "distinct expert rows"
        eq(got, exp, f"ll combine of the {kind} (sampled tokens, microbatch {t0}){what}")


def _ll_full(wl):
    R, E, K, T, H, cap = wl.R, wl.E, wl.K, wl.T, wl.H, wl.ll_cap
    L = E // R
    idx, w = inputs.make_routing(wl, 0)
    x = inputs.make_x(wl, 0, device="cuda")
    xf = x.view(R * T, H)
    buf = LLBuffer(R, E, K, T, H, cap)
    idxd, wd = idx.cuda(), w.cuda()
    out = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
    out_y = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
    pk = buf.alloc_packed()
    y_rand = inputs.random_rows(R * L * R * cap, H, seed=77, device="cuda").view(pk["packed_x"].shape)
    q = _oracle_fp8_rows(xf)                    # every token's codes and scales, by the oracle
    rng = np.random.default_rng(11)
    for t0 in range(0, T, cap):
        n = min(cap, T - t0)
        buf.dispatch(x, idxd, t0, n, out=pk)
        buf.check()
        y_ll = _identity_y(pk, R)
        buf.combine(y_ll, idxd, wd, pk, t0, n, out=out)
        buf.combine(y_rand, idxd, wd, pk, t0, n, out=out_y)
        buf.check()
        _check_ll_microbatch_full(pk, [(out, y_ll, True), (out_y, y_rand, False)], xf, q, idx, w, R, E, K, T, H,
                                  cap, t0, n, rng)
        del y_ll


def test_decode_ll_full():
    _ll_full(inputs.WORKLOADS["decode"])


def test_skewed_ll_full_microbatches():
    _ll_full(inputs.WORKLOADS["skewed"])


def test_prefill_full_fp8_one_pass():
    """The FP8 dispatches at the prefill size, in the bench's launch
    configuration: every row of the one-pass forms (into the permuted layout
    and into the receive layout) and of the two-pass form (quantise, then the
    fused FP8 dispatch) equals the oracle's quantisation of the source token
    the oracle assigned to that row."""
    wl = inputs.WORKLOADS["prefill"]
    R, E, K, T, H, C = wl.R, wl.E, wl.K, wl.T, wl.H, wl.num_channels
    idx, w = inputs.make_routing(wl, 0)
    x = inputs.make_x(wl, 0, device="cuda")
    xf = x.view(R * T, H)
    ctx = Context(R, E, K, T, H, num_channels=C)
    idxd, wd = idx.cuda(), w.cuda()
    h = ctx.notify_dispatch(idxd, ctx.get_dispatch_layout(idxd))
    n_def = H + H // 32
    # the oracle's row assignment (positions do not depend on H: 8-channel stand-in)
    o_lay = orc.layout(idx, R, E)
    o_note = orc.notify(o_lay, R, E, T, C)
    o_disp = orc.dispatch(np.zeros((R, T, 8), np.uint16), idx, w, o_note, R, E)
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    recv_tok = o_disp["recv_src_rank"].astype(np.int64) * T + o_disp["recv_src_idx"]
    perm_tok = recv_tok[o_perm["perm_src_row"]]
    q = _oracle_fp8_rows(xf)
    one = ctx.dispatch_permuted_quant(x, idxd, wd, h)
    ctx.check()
    _rows_equal(one["permuted_xq"][:, :n_def], q, perm_tok, "permuted_xq (one pass)")
    eq(one["perm_src_token"], perm_tok.astype(np.int32), "perm_src_token (one pass)")
    del one
    xq = ctx.quantize_fp8(x)
    _rows_equal(xq[:, :n_def], q, np.arange(R * T), "quantised rows")
    two = ctx.dispatch_permuted_fp8(xq, idxd, wd, h)
    ctx.check()
    _rows_equal(two["permuted_xq"][:, :n_def], q, perm_tok, "permuted_xq (two passes)")
    del two
    recv = ctx.dispatch_quant(x, idxd, wd, h)
    ctx.check()
    _rows_equal(recv["recv_xq"][:, :n_def], q, recv_tok, "recv_xq (one pass)")
    for k in ("recv_src_rank", "recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        eq(recv[k], o_disp[k], k)


def _combine_sampled(out, xf, idx, w, R, E, K, T, H, what):
    """Identity-expert combine of sampled tokens against the oracle's
    sub-problem (every entry of a token reads the token's own row)."""
    rng = np.random.default_rng(13)
    g = rng.choice(R * T, size=min(N_SAMPLES, R * T), replace=False)
    gd = torch.from_numpy(g).cuda()
    xs = bits(xf.index_select(0, gd))
    exp = _combine_sub_problem(np.repeat(xs[:, None, :], K, axis=1), idx.numpy().reshape(R * T, K),
                               w.numpy().reshape(R * T, K), g, R, E, K, False, 1)
    eq(bits(out.view(R * T, H).index_select(0, gd)), exp, what)


def test_prefill_full_expert_aligned():
    """The permute into 128-row aligned expert blocks at the prefill size (the
    bench's expert_aligned leg): the handle's offsets, every pair's position and
    row, and the combine reading the aligned layout."""
    wl = inputs.WORKLOADS["prefill"]
    R, E, K, T, H, C = wl.R, wl.E, wl.K, wl.T, wl.H, wl.num_channels
    align = 128
    idx, w = inputs.make_routing(wl, 0)
    x = inputs.make_x(wl, 0, device="cuda")
    xf = x.view(R * T, H)
    ctx = Context(R, E, K, T, H, num_channels=C, expert_alignment=align)
    idxd, wd = idx.cuda(), w.cuda()
    h = ctx.notify_dispatch(idxd, ctx.get_dispatch_layout(idxd))
    recv = ctx.dispatch(x, idxd, wd, h)
    perm = ctx.permute(h, recv)
    out = ctx.combine(h, perm["permuted_x"], idxd, wd)
    ctx.check()
    torch.cuda.synchronize()
    o_note = orc.notify(orc.layout(idx, R, E), R, E, T, C, align=align)
    for k in ("num_recv_per_expert", "expert_offsets", "perm_rank_base"):
        eq(h[k], o_note[k], k)
    o_disp = orc.dispatch(np.zeros((R, T, 8), np.uint16), idx, w, o_note, R, E)
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    eq(h["perm_pos"], o_perm["perm_pos"], "perm_pos")
    psr = o_perm["perm_src_row"]
    used = np.nonzero(psr >= 0)[0]
    assert perm["permuted_x"].shape[0] == len(psr)
    eq(perm["perm_src_row"].cpu().numpy()[used], psr[used], "perm_src_row (pairs' rows)")
    src_tok = o_disp["recv_src_rank"].astype(np.int64) * T + o_disp["recv_src_idx"]
    _rows_equal(perm["permuted_x"], xf, src_tok[psr[used]], "permuted_x (aligned)", got_rows=used)
    _combine_sampled(out, xf, idx, w, R, E, K, T, H, "combine of the aligned layout (sampled tokens)")


def test_prefill_full_no_wait_graph():
    """The prefill step without the host wait, captured in one CUDA graph and
    replayed (the bench's graph leg): worst-case buffers, row totals read on
    the device; the handle, every received and permuted row, and sampled
    combine tokens equal the oracle's."""
    wl = inputs.WORKLOADS["prefill"]
    R, E, K, T, H, C = wl.R, wl.E, wl.K, wl.T, wl.H, wl.num_channels
    idx, w = inputs.make_routing(wl, 0)
    x = inputs.make_x(wl, 0, device="cuda")
    xf = x.view(R * T, H)
    ctx = Context(R, E, K, T, H, num_channels=C)
    idxd, wd = idx.cuda(), w.cuda()
    rmax, pmax, _ = ctx.max_rows
    recv = ctx.alloc_recv(rmax)
    perm = dict(permuted_x=torch.empty(pmax, H, dtype=torch.bfloat16, device="cuda"),
                perm_src_row=torch.empty(pmax, dtype=torch.int32, device="cuda"))
    out = torch.empty(R, T, H, dtype=torch.bfloat16, device="cuda")
    lay = {k: v for k, v in ctx.get_dispatch_layout(idxd).items()}
    h = ctx.alloc_handle()

    def step():
        ctx.get_dispatch_layout(idxd, out=lay)
        ctx.notify_dispatch(idxd, lay, handle=h, wait=False)
        ctx.dispatch(x, idxd, wd, h, out=recv)
        ctx.permute(h, recv, out=perm)
        ctx.combine(h, perm["permuted_x"], idxd, wd, out=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # once outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    recv["recv_x"].zero_()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    torch.cuda.synchronize()
    ctx.check()
    o_note = orc.notify(orc.layout(idx, R, E), R, E, T, C)
    for k in ("recv_count", "num_recv_tokens", "recv_offsets", "rank_base", "num_recv_per_expert",
              "expert_offsets", "perm_rank_base", "channel_prefix_matrix", "send_pos"):
        eq(h[k], o_note[k], k)
    nr, npm = int(o_note["rank_base"][R]), int(o_note["perm_rank_base"][R])
    o_disp = orc.dispatch(np.zeros((R, T, 8), np.uint16), idx, w, o_note, R, E)
    for k in ("recv_src_rank", "recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        eq(recv[k][:nr], o_disp[k], k)
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    eq(h["perm_pos"], o_perm["perm_pos"], "perm_pos")
    eq(perm["perm_src_row"][:npm], o_perm["perm_src_row"], "perm_src_row")
    src_tok = o_disp["recv_src_rank"].astype(np.int64) * T + o_disp["recv_src_idx"]
    _rows_equal(recv["recv_x"][:nr], xf, src_tok, "recv_x (graph replay)")
    _rows_equal(perm["permuted_x"][:npm], xf, src_tok[o_perm["perm_src_row"]], "permuted_x (graph replay)")
    _combine_sampled(out, xf, idx, w, R, E, K, T, H, "combine (graph replay, sampled tokens)")


def test_decode_ll_full_graph_and_two_streams():
    """The decode layer as the bench also times it: replayed from a CUDA graph,
    and two microbatches (two buffers, different tokens) sent, received and
    combined on two streams at once.  Every message and sampled combine
    tokens of each equal the oracle's."""
    wl = inputs.WORKLOADS["decode"]
    R, E, K, T, H, cap = wl.R, wl.E, wl.K, wl.T, wl.H, wl.ll_cap
    L = E // R
    rng = np.random.default_rng(19)
    lanes = []
    for seed in (0, 1):
        idx, w = inputs.make_routing(wl, seed)
        x = inputs.make_x(wl, seed, device="cuda")
        buf = LLBuffer(R, E, K, T, H, cap)
        pk = buf.alloc_packed()
        y = inputs.random_rows(R * L * R * cap, H, seed=31 + seed, device="cuda").view(pk["packed_x"].shape)
        out = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
        lanes.append(dict(idx=idx, w=w, x=x, idxd=idx.cuda(), wd=w.cuda(), buf=buf, pk=pk, y=y, out=out,
                          q=_oracle_fp8_rows(x.view(R * T, H))))
    # one lane as a CUDA graph, replayed
    a = lanes[0]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        a["buf"].dispatch(a["x"], a["idxd"], out=a["pk"])
        a["buf"].combine(a["y"], a["idxd"], a["wd"], a["pk"], out=a["out"])
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        a["buf"].dispatch(a["x"], a["idxd"], out=a["pk"])
        a["buf"].combine(a["y"], a["idxd"], a["wd"], a["pk"], out=a["out"])
    a["out"].zero_()
    a["pk"]["packed_recv_count"].fill_(-5)
    g.replay()
    torch.cuda.synchronize()
    a["buf"].check()
    _check_ll_microbatch_full(a["pk"], [(a["out"], a["y"], False)], a["x"].view(R * T, H), a["q"], a["idx"], a["w"],
                              R, E, K, T, H, cap, 0, T, rng, " (graph replay)")
    del g
    # both lanes on two streams at once
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    main = torch.cuda.current_stream()
    for ln in lanes:
        ln["out"].zero_()
    for st, ln in zip(streams, lanes):
        st.wait_stream(main)
        with torch.cuda.stream(st):
            ln["buf"].dispatch(ln["x"], ln["idxd"], out=ln["pk"])
            ln["buf"].combine(ln["y"], ln["idxd"], ln["wd"], ln["pk"], out=ln["out"])
    for st in streams:
        main.wait_stream(st)
    torch.cuda.synchronize()
    for i, ln in enumerate(lanes):
        ln["buf"].check()
        _check_ll_microbatch_full(ln["pk"], [(ln["out"], ln["y"], False)], ln["x"].view(R * T, H), ln["q"], ln["idx"],
                                  ln["w"], R, E, K, T, H, cap, 0, T, rng, f" (stream {i} of two)")
