"""Failure detection without a GPU fault: bad inputs are caught on the host or
flagged by the kernels' own checks; a wait on a count slot that nothing
writes runs out (short limit) and comes back as EP_ERR_TIMEOUT, after which
the context keeps working."""
import time

import pytest
import torch

from combine_get_dispatch_histograms_gb300 import Context, EpError, LLBuffer, inputs

pytestmark = pytest.mark.gpu


def test_ll_receive_times_out_when_nothing_was_sent():
    R, E, K, T, H, cap = 4, 8, 2, 8, 128, 8
    buf = LLBuffer(R, E, K, T, H, cap)
    buf.set_wait_timeout_us(20_000)  # 20 ms
    pk = buf.alloc_packed()
    t = time.time()
    buf.recv(pk)  # count slots of the current buffer still hold the sentinel
    with pytest.raises(EpError) as e:
        buf.check()
    assert e.value.status == "EP_ERR_TIMEOUT"
    assert time.time() - t < 30
    assert (pk["packed_recv_count"] == 0).all()
    # the buffer and the GPU stay usable: a real dispatch now works
    idx = inputs.random_topk(R, E, K, T, 0)
    x = inputs.random_x(R, T, H, 0)
    pk = buf.dispatch(x.cuda(), idx.cuda())
    buf.check()
    assert int(pk["packed_recv_count"].sum()) == int((idx >= 0).sum())


def test_invalid_topk_is_reported():
    R, E, K, T, H = 4, 8, 2, 20, 64
    idx = inputs.random_topk(R, E, K, T, 1)
    idx[2, 5, 1] = 8    # == E
    idx[0, 0, 0] = -7
    ctx = Context(R, E, K, T, H, num_channels=2)
    lay = ctx.get_dispatch_layout(idx.cuda())
    with pytest.raises(EpError) as e:
        ctx.notify_dispatch(idx.cuda(), lay)
    assert e.value.status == "EP_ERR_INVALID_INPUT"
    with pytest.raises(EpError):
        ctx.check()
    ctx.check()  # cleared
    # valid entries of the bad tokens are still counted
    assert int(lay["num_tokens_per_expert"].sum()) == int(((idx >= 0) & (idx < E)).sum())


def test_host_side_argument_checks():
    R, E, K, T, H = 4, 8, 2, 20, 64
    idx = inputs.random_topk(R, E, K, T, 2).cuda()
    x = inputs.random_x(R, T, H, 2).cuda()
    w = inputs.random_weights(R, T, K, 2).cuda()
    ctx = Context(R, E, K, T, H, num_channels=2)
    h = ctx.notify_dispatch(idx, ctx.get_dispatch_layout(idx))
    # recv buffers one row short
    small = ctx.alloc_recv(h.num_recv_rows - 1)
    with pytest.raises(EpError) as e:
        ctx.dispatch(x, idx, w, h, out=small)
    assert e.value.status == "EP_ERR_CAPACITY"
    # misaligned x
    xm = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + x.numel()].view_as(x)
    with pytest.raises(EpError) as e:
        ctx.dispatch(xm, idx, w, h)
    assert e.value.status == "EP_ERR_INVALID_ARG"
    # hierarchical entry points on a flat context
    with pytest.raises(EpError):
        ctx.combine(h, x.view(-1, H), idx, w, hier=True)


def test_ll_capacity_checks():
    R, E, K, T, H, cap = 2, 4, 2, 8, 128, 4
    buf = LLBuffer(R, E, K, T, H, cap)
    idx = torch.zeros(R, T, K, dtype=torch.int64)
    x = inputs.random_x(R, T, H, 3)
    with pytest.raises(EpError) as e:
        buf.dispatch(x.cuda(), idx.cuda(), 0, T)  # microbatch larger than the cap
    assert e.value.status == "EP_ERR_CAPACITY"
    # duplicate experts in a token overflow a region inside the cap: flagged on the device
    idx[:, :, :] = 1
    buf.dispatch(x.cuda(), idx.cuda(), 0, cap)
    with pytest.raises(EpError) as e:
        buf.check()
    assert e.value.status == "EP_ERR_CAPACITY"
