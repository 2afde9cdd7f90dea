"""Expert-aligned permuted layout on the GPU against the oracle: the handle
(expert offsets rounded to the alignment, permuted totals with padding,
perm_pos), every pair's row of the permute, the fused dispatch and its FP8
form, and the combine reading the aligned layout; padding rows are not
compared (they are not written).  Also with the no-wait notify and the
hierarchical path."""
import numpy as np
import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, inputs
from parity_util import bits, eq

pytestmark = pytest.mark.gpu


def _check(R, E, K, T, H, C, mask_p, align, seed, nodes=1, hier=False, wait=True):
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    ctx = Context(R, E, K, T, H, num_channels=C, num_nodes=nodes, expert_alignment=align)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    lay = ctx.get_dispatch_layout(idxd, nodes=nodes > 1)
    h = ctx.notify_dispatch(idxd, lay, wait=wait)
    if wait:
        recv = ctx.dispatch_hier(xd, idxd, wd, h) if hier else ctx.dispatch(xd, idxd, wd, h)
        perm = ctx.permute(h, recv)
        fused = ctx.dispatch_permuted(xd, idxd, wd, h)
    else:
        rmax, pmax, smax = ctx.max_rows
        recv = ctx.alloc_recv(rmax)
        if hier:
            st = dict(staging=torch.empty(smax, H, dtype=torch.bfloat16, device="cuda"),
                      stage_src_rank=torch.empty(smax, dtype=torch.int32, device="cuda"),
                      stage_src_idx=torch.empty(smax, dtype=torch.int32, device="cuda"))
            ctx.dispatch_hier(xd, idxd, wd, h, out=recv, staging=st)
        else:
            ctx.dispatch(xd, idxd, wd, h, out=recv)
        perm = ctx.permute(h, recv, out=dict(permuted_x=torch.empty(pmax, H, dtype=torch.bfloat16, device="cuda"),
                                             perm_src_row=torch.empty(pmax, dtype=torch.int32, device="cuda")))
        fused = ctx.dispatch_permuted(xd, idxd, wd, h, out=dict(
            permuted_x=torch.empty(pmax, H, dtype=torch.bfloat16, device="cuda"),
            perm_src_token=torch.empty(pmax, dtype=torch.int32, device="cuda"),
            perm_weight=torch.empty(pmax, dtype=torch.float32, device="cuda")))
    out = ctx.combine(h, perm["permuted_x"], idxd, wd, hier=hier)
    ctx.check()
    torch.cuda.synchronize()

    o_lay = orc.layout(idx, R, E, num_nodes=nodes if nodes > 1 else 0)
    o_note = orc.notify(o_lay, R, E, T, C, align=align)
    for k in ("num_recv_per_expert", "expert_offsets", "perm_rank_base", "rank_base", "send_pos"):
        eq(h[k], o_note[k], k)
    P = int(o_note["perm_rank_base"][R])
    if wait:
        assert h.num_perm_rows == P
        assert perm["permuted_x"].shape[0] == P
    o_disp = orc.dispatch(x, idx, w, o_note, R, E)
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    eq(h["perm_pos"], o_perm["perm_pos"], "perm_pos")
    used = o_perm["perm_src_row"] >= 0
    eq(bits(perm["permuted_x"][:P])[used], o_perm["permuted_x"][used], "permuted_x (pair rows)")
    eq(bits(perm["perm_src_row"][:P])[used], o_perm["perm_src_row"][used], "perm_src_row (pair rows)")
    eq(bits(fused["permuted_x"][:P])[used], o_perm["permuted_x"][used], "fused permuted_x (pair rows)")
    src_tok = (o_disp["recv_src_rank"].astype(np.int64) * T + o_disp["recv_src_idx"]).astype(np.int32)
    eq(bits(fused["perm_src_token"][:P])[used], src_tok[o_perm["perm_src_row"][used]], "perm_src_token")
    if hier:
        o_out = orc.combine_hier(o_perm["permuted_x"], o_perm["perm_pos"], idx, w, R, E, nodes)
    else:
        o_out = orc.combine(o_perm["permuted_x"], o_perm["perm_pos"], idx, w, R, E, "ord32")
    eq(out, o_out, "combine on the aligned layout")
    return ctx, h, idxd, wd, xd, o_perm, used, P


@pytest.mark.parametrize("R,E,K,T,H,C,mask_p,align,seed", [
    (4, 16, 4, 333, 64, 5, 0.3, 8, 1),
    (8, 256, 8, 300, 256, 8, 0.0, 128, 2),
    (4, 8, 2, 100, 64, 2, 0.0, 3, 3),         # alignment not a power of two
    (4, 8, 2, 60, 64, 2, 1.0, 16, 4),         # all masked: no rows at all
    (2, 64, 2, 5, 64, 2, 0.0, 64, 5),         # most experts empty
])
def test_aligned_normal(R, E, K, T, H, C, mask_p, align, seed):
    _check(R, E, K, T, H, C, mask_p, align, seed)


def test_aligned_no_wait():
    _check(8, 64, 8, 200, 128, 4, 0.05, 32, 6, wait=False)


def test_aligned_hier():
    _check(8, 32, 4, 300, 64, 4, 0.05, 16, 7, nodes=2, hier=True)


def test_aligned_fp8_rows():
    R, E, K, T, H, C, align = 4, 16, 4, 150, 256, 4, 64
    ctx, h, idxd, wd, xd, o_perm, used, P = _check(R, E, K, T, H, C, 0.1, align, 8)
    xq = ctx.quantize_fp8(xd)
    recvq = ctx.dispatch_fp8(xq, idxd, wd, h)
    permq = ctx.permute_fp8(h, recvq)
    fusedq = ctx.dispatch_permuted_fp8(xq, idxd, wd, h)
    ctx.check()
    xq_np = bits(xq)
    src = o_perm["perm_src_row"][used]
    # the FP8 rows of the recv rows the oracle placed, row for row
    recv_rows = bits(recvq["recv_xq"])
    eq(bits(permq["permuted_xq"][:P])[used], recv_rows[src], "permuted FP8 rows")
    tok = bits(fusedq["perm_src_token"][:P])[used]
    eq(bits(fusedq["permuted_xq"][:P])[used], xq_np[tok], "fused FP8 rows")


def test_fresh_context_has_alignment_one_and_nothing_notified():
    """A fresh context starts with expert alignment 1 (no padding) and with
    zero known rows, so a copy launched before any notify does nothing."""
    R, E, K, T, H = 4, 8, 2, 16, 128
    ctx = Context(R, E, K, T, H)
    assert ctx.lib.ep_ctx_expert_alignment(ctx._ctx) == 1
    ctx.set_expert_alignment(16)
    assert ctx.lib.ep_ctx_expert_alignment(ctx._ctx) == 16
    ctx.set_expert_alignment(1)
    assert ctx.lib.ep_ctx_expert_alignment(ctx._ctx) == 1
    # the default alignment gives the oracle's unpadded offsets
    idx = inputs.random_topk(R, E, K, T, 3, 0.1)
    fresh = Context(R, E, K, T, H)
    lay = fresh.get_dispatch_layout(idx.cuda())
    h = fresh.notify_dispatch(idx.cuda(), lay)
    torch.cuda.synchronize()
    o_note = orc.notify(orc.layout(idx, R, E), R, E, T, 8)
    for k in ("expert_offsets", "perm_rank_base"):
        eq(h[k], o_note[k], k)
