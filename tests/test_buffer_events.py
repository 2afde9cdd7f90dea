"""The event-driven Buffer protocol: work runs on the communication stream
and gives the direct calls' results, synchronously (the compute stream waits)
and asynchronously (the caller waits on the returned event)."""
import pytest
import torch

from combine_get_dispatch_histograms_gb300 import Context, inputs
from combine_get_dispatch_histograms_gb300.buffer import Buffer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("async_finish", [False, True])
def test_buffer_matches_direct_calls(async_finish):
    R, E, K, T, H, C = 4, 16, 4, 300, 128, 4
    idx = inputs.random_topk(R, E, K, T, 50, 0.1).cuda()
    x = inputs.random_x(R, T, H, 50).cuda()
    w = inputs.random_weights(R, T, K, 50).cuda()
    ctx = Context(R, E, K, T, H, num_channels=C)
    # direct
    lay0 = ctx.get_dispatch_layout(idx)
    h0 = ctx.notify_dispatch(idx, lay0)
    recv0 = ctx.dispatch(x, idx, w, h0)
    perm0 = ctx.permute(h0, recv0)
    out0 = ctx.combine(h0, perm0["permuted_x"], idx, w)
    torch.cuda.synchronize()
    # through the Buffer, on its own stream
    buf = Buffer(ctx)
    lay, ev = buf.get_dispatch_layout(idx, async_finish=async_finish)
    res = buf.dispatch(x, idx, w, layout=lay, previous_event=ev, async_finish=async_finish)
    perm, ev2 = buf.permute(res, previous_event=res.event, async_finish=async_finish)
    if async_finish:
        ev2.current_stream_wait()
    y = perm["permuted_x"] * 1  # the "expert" runs on the compute stream
    out, ev3 = buf.combine(res, y, idx, w, async_finish=async_finish)
    if async_finish:
        ev3.current_stream_wait()
    torch.cuda.synchronize()
    ctx.check()
    for k in lay0:
        assert torch.equal(lay[k], lay0[k]), k
    for k in ("recv_x", "recv_src_rank", "recv_src_idx"):
        assert torch.equal(res.recv[k], recv0[k]), k
    assert torch.equal(perm["permuted_x"].view(torch.int16), perm0["permuted_x"].view(torch.int16))
    assert torch.equal(out.view(torch.int16), out0.view(torch.int16))


def test_buffer_hierarchical():
    import numpy as np
    import oracle as orc
    from parity_util import eq
    R, E, K, T, H, C, N = 8, 32, 4, 200, 64, 4, 2
    idx_c = inputs.random_topk(R, E, K, T, 51, 0.05)
    x_c, w_c = inputs.random_x(R, T, H, 51), inputs.random_weights(R, T, K, 51)
    ctx = Context(R, E, K, T, H, num_channels=C, num_nodes=N)
    buf = Buffer(ctx)
    idx, x, w = idx_c.cuda(), x_c.cuda(), w_c.cuda()
    res = buf.dispatch(x, idx, w)
    perm, _ = buf.permute(res)
    out, _ = buf.combine(res, perm["permuted_x"], idx, w)
    torch.cuda.synchronize()
    ctx.check()
    o_lay = orc.layout(idx_c, R, E, num_nodes=N)
    o_note = orc.notify(o_lay, R, E, T, C)
    o_disp = orc.dispatch(x_c, idx_c, w_c, o_note, R, E)
    o_perm = orc.permute(idx_c, o_disp["recv_x"], o_note, R, E)
    eq(out, orc.combine_hier(o_perm["permuted_x"], o_perm["perm_pos"], idx_c, w_c, R, E, N), "combine (hier)")
