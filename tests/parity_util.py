"""Helpers of the GPU parity tests: run the CUDA path through the binding and
the oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, LLBuffer, inputs


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def eq(got, exp, what: str):
    got = bits(got) if isinstance(got, torch.Tensor) else np.asarray(got)
    exp = np.asarray(exp)
    assert got.shape == exp.shape, f"{what}: shape {got.shape} != {exp.shape}"
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {i}: got {got[i]} expected {exp[i]}")


def run_gpu_normal(R, E, K, T, H, C, x, idx, w, nodes=1, hier=False, dev="cuda"):
    ctx = Context(R, E, K, T, H, num_channels=C, num_nodes=nodes)
    xd, idxd, wd = x.to(dev), idx.to(dev), w.to(dev)
    lay = ctx.get_dispatch_layout(idxd, nodes=nodes > 1)
    h = ctx.notify_dispatch(idxd, lay)
    if hier:
        recv = ctx.dispatch_hier(xd, idxd, wd, h)
    else:
        recv = ctx.dispatch(xd, idxd, wd, h)
    perm = ctx.permute(h, recv)
    out = ctx.combine(h, perm["permuted_x"], idxd, wd, hier=hier)
    ctx.check()
    torch.cuda.synchronize()
    return ctx, lay, h, recv, perm, out


def compare_normal(R, E, K, T, H, C, x, idx, w, nodes=1, hier=False):
    ctx, lay, h, recv, perm, out = run_gpu_normal(R, E, K, T, H, C, x, idx, w, nodes, hier)
    o_lay = orc.layout(idx, R, E, num_nodes=nodes if nodes > 1 else 0)
    for k in ("num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank"):
        eq(lay[k], o_lay[k], k)
    if nodes > 1:
        eq(lay["num_tokens_per_node"], o_lay["num_tokens_per_node"], "num_tokens_per_node")
        eq(lay["is_token_in_node"], o_lay["is_token_in_node"], "is_token_in_node")
    o_note = orc.notify(o_lay, R, E, T, C)
    for k in ("recv_count", "num_recv_tokens", "recv_offsets", "rank_base", "num_recv_per_expert",
              "expert_offsets", "perm_rank_base", "channel_prefix_matrix", "send_pos"):
        eq(h[k], o_note[k], k)
    assert list(h.host_num_recv_tokens) == list(o_note["num_recv_tokens"])
    assert h.num_recv_rows == int(o_note["rank_base"][R])
    assert h.num_perm_rows == int(o_note["perm_rank_base"][R])
    o_disp = orc.dispatch(x, idx, w, o_note, R, E)
    for k in ("recv_x", "recv_src_rank", "recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        eq(recv[k], o_disp[k], k)
    if hier:
        sb, sp = orc.hier_stage_pos(o_lay, R, T, nodes)
        eq(h["stage_base"], sb, "stage_base")
        eq(h["stage_pos"], sp, "stage_pos")
        o_st = orc.hier_dispatch(x, o_lay, o_note, sb, sp, R, nodes)
        eq(recv["staging"], o_st["staging"], "staging")
        eq(recv["stage_src_rank"], o_st["stage_src_rank"], "stage_src_rank")
        eq(recv["stage_src_idx"], o_st["stage_src_idx"], "stage_src_idx")
        eq(recv["recv_x"], o_st["recv_x"], "recv_x (staged)")
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    eq(h["perm_pos"], o_perm["perm_pos"], "perm_pos")
    eq(perm["permuted_x"], o_perm["permuted_x"], "permuted_x")
    eq(perm["perm_src_row"], o_perm["perm_src_row"], "perm_src_row")
    # fused dispatch straight into the permuted layout: the same rows
    fused = ctx.dispatch_permuted(x.cuda(), idx.cuda(), w.cuda(), h)
    ctx.check()
    eq(fused["permuted_x"], o_perm["permuted_x"], "permuted_x (fused dispatch)")
    pp = o_perm["perm_pos"]
    P = int((pp >= 0).sum())
    exp_tok = np.full(P, -1, np.int32)
    exp_w = np.zeros(P, np.float32)
    wn = w.numpy() if hasattr(w, "numpy") else np.asarray(w)
    for s_, t_, k_ in zip(*np.nonzero(pp >= 0)):
        exp_tok[pp[s_, t_, k_]] = s_ * T + t_
        exp_w[pp[s_, t_, k_]] = wn[s_, t_, k_]
    eq(fused["perm_src_token"], exp_tok, "perm_src_token")
    eq(fused["perm_weight"], exp_w, "perm_weight")
    if hier:
        o_out = orc.combine_hier(o_perm["permuted_x"], o_perm["perm_pos"], idx, w, R, E, nodes)
    else:
        o_out = orc.combine(o_perm["permuted_x"], o_perm["perm_pos"], idx, w, R, E, "ord32")
    eq(out, o_out, "combine (fp32 order)")
    check_tolerance(out, orc.combine(o_perm["permuted_x"], o_perm["perm_pos"], idx, w, R, E, "ref64"))
    # an expert output with a different row for every permuted row: a combine
    # that reads another pair's row of the same token changes the bits
    y = inputs.random_rows(int(o_perm["permuted_x"].shape[0]), H, seed=int(T) * 131 + R)
    out_y = ctx.combine(h, y.cuda(), idx.cuda(), w.cuda(), hier=hier)
    ctx.check()
    if hier:
        o_y = orc.combine_hier(y, o_perm["perm_pos"], idx, w, R, E, nodes)
    else:
        o_y = orc.combine(y, o_perm["perm_pos"], idx, w, R, E, "ord32")
    eq(out_y, o_y, "combine of distinct expert rows (fp32 order)")
    check_tolerance(out_y, orc.combine(y, o_perm["perm_pos"], idx, w, R, E, "ref64"))
    return ctx


def check_tolerance(out: torch.Tensor, ref64_bits: np.ndarray):
    """max-abs 1e-2 and relative 4e-3 against the fp64 reference, read as
    |got - ref| <= 1e-2 + 4e-3 |ref|, except where the two differ by one bf16
    ulp (an fp32 sum that landed on the other side of a bf16 midpoint)."""
    got = out.detach().float().cpu().numpy()
    ref = torch.from_numpy(ref64_bits.view(np.int16)).view(torch.bfloat16).float().numpy().reshape(got.shape)
    diff = np.abs(got - ref)
    ok = diff <= 1e-2 + 4e-3 * np.abs(ref)
    one_ulp = diff <= np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
    assert (ok | one_ulp).all(), f"{(~(ok | one_ulp)).sum()} elements outside the tolerance"
    return int((~ok).sum())


def run_gpu_ll(R, E, K, T, H, cap, x, idx, microbatches):
    buf = LLBuffer(R, E, K, T, H, cap)
    xd, idxd = x.cuda(), idx.cuda()
    outs = []
    for t0, n in microbatches:
        pk = buf.dispatch(xd, idxd, t0, n)
        torch.cuda.synchronize()
        outs.append({k: v.clone() for k, v in pk.items()})
    buf.check()
    return buf, outs


def check_ll_microbatch_equal(pk, sent, o_pk, R, E, T, cap, t0=0, n=None):
    """The low-latency send's slots and the receive's packed outputs against
    the oracle's for the microbatch [t0, t0 + n): slots, counts, layout
    ranges and every packed message (codes, scales, source)."""
    n = T - t0 if n is None else n
    L = E // R
    eq(pk["slot"][:, t0:t0 + n], sent["slot"][:, t0:t0 + n], "slot")
    eq(pk["packed_recv_count"], o_pk["packed_recv_count"], "packed_recv_count")
    eq(pk["layout_range"], o_pk["layout_range"], "layout_range")
    px, ps, pi = bits(pk["packed_x"]), bits(pk["packed_scales"]), bits(pk["packed_src_info"])
    for d in range(R):
        for l in range(L):
            c = int(o_pk["packed_recv_count"][d, l])
            eq(px[d, l, :c], o_pk["packed_x"][d, l, :c], f"packed_x[{d},{l}]")
            eq(ps[d, l, :c], o_pk["packed_scales"][d, l, :c], f"packed_scales[{d},{l}]")
            eq(pi[d, l, :c], o_pk["packed_src_info"][d, l, :c], f"packed_src_info[{d},{l}]")
