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


def test_one_pass_fp8_capacity_and_arguments():
    """The one-pass FP8 dispatches: a buffer one row short is caught on the host
    after a waiting notify and flagged on the device after a no-wait one; a
    hidden size that is not a multiple of 128 is refused."""
    R, E, K, T, H = 4, 16, 4, 64, 256
    idx = inputs.random_topk(R, E, K, T, 60).cuda()
    x = inputs.random_x(R, T, H, 60).cuda()
    w = inputs.random_weights(R, T, K, 60).cuda()
    ctx = Context(R, E, K, T, H, num_channels=2)
    h = ctx.notify_dispatch(idx, ctx.get_dispatch_layout(idx))
    rq = ctx.fp8_row_bytes
    short = dict(permuted_xq=torch.empty(h.num_perm_rows - 1, rq, dtype=torch.uint8, device="cuda"),
                 perm_src_token=torch.empty(h.num_perm_rows - 1, dtype=torch.int32, device="cuda"),
                 perm_weight=torch.empty(h.num_perm_rows - 1, dtype=torch.float32, device="cuda"))
    with pytest.raises(EpError) as e:
        ctx.dispatch_permuted_quant(x, idx, w, h, out=short)
    assert e.value.status == "EP_ERR_CAPACITY"
    h2 = ctx.notify_dispatch(idx, ctx.get_dispatch_layout(idx), wait=False)
    ctx.dispatch_permuted_quant(x, idx, w, h2, out=short)
    with pytest.raises(EpError) as e:
        ctx.check()
    assert e.value.status == "EP_ERR_CAPACITY"
    rows = h.num_recv_rows - 1
    short_recv = dict(recv_xq=torch.empty(rows, rq, dtype=torch.uint8, device="cuda"),
                      recv_src_rank=torch.empty(rows, dtype=torch.int32, device="cuda"),
                      recv_src_idx=torch.empty(rows, dtype=torch.int32, device="cuda"),
                      recv_topk_idx=torch.empty(rows, K, dtype=torch.int32, device="cuda"),
                      recv_topk_weights=torch.empty(rows, K, dtype=torch.float32, device="cuda"))
    ctx.dispatch_quant(x, idx, w, h2, out=short_recv)
    with pytest.raises(EpError) as e:
        ctx.check()
    assert e.value.status == "EP_ERR_CAPACITY"
    odd = Context(R, E, K, T, 136, num_channels=2)
    x136 = inputs.random_x(R, T, 136, 60).cuda()
    h3 = odd.notify_dispatch(idx, odd.get_dispatch_layout(idx))
    with pytest.raises(EpError) as e:
        odd.dispatch_quant(x136, idx, w, h3, out=short_recv)
    assert e.value.status == "EP_ERR_INVALID_ARG"


def test_layout_notify_argument_checks():
    R, E, K, T = 8, 16, 2, 20
    idx = inputs.random_topk(R, E, K, T, 61).cuda()
    flat = Context(R, E, K, T, 64, num_channels=2)
    lay = dict(num_tokens_per_expert=torch.empty(R, E, dtype=torch.int32, device="cuda"),
               num_tokens_per_rank=torch.empty(R, R, dtype=torch.int32, device="cuda"),
               is_token_in_rank=torch.empty(R, T, R, dtype=torch.uint8, device="cuda"),
               num_tokens_per_node=torch.empty(R, 2, dtype=torch.int32, device="cuda"),
               is_token_in_node=torch.empty(R, T, 2, dtype=torch.uint8, device="cuda"))
    h = flat.alloc_handle()
    with pytest.raises(EpError) as e:  # node outputs on a flat context
        check_raw(flat, idx, lay, h)
    assert e.value.status == "EP_ERR_INVALID_ARG"


def check_raw(ctx, idx, lay, h):
    """ep_layout_notify called with node outputs given (bypassing the binding's choice)."""
    import ctypes
    from combine_get_dispatch_histograms_gb300 import _lib
    p = lambda t: t.data_ptr()
    rc = ctx.lib.ep_layout_notify(ctx._ctx, p(idx), p(lay["num_tokens_per_expert"]), p(lay["num_tokens_per_rank"]),
                                  p(lay["is_token_in_rank"]), p(lay["num_tokens_per_node"]),
                                  p(lay["is_token_in_node"]), ctypes.byref(h.c_struct()), ctx._host_recv, None, None,
                                  torch.cuda.current_stream().cuda_stream)
    _lib.check("ep_layout_notify", rc)


def test_ll_signal_wait_trace():
    """The receive's signal-wait trace: about the time limit when nothing was
    sent, small waits once the counts are published."""
    R, E, K, T, H, cap = 4, 8, 2, 8, 128, 8
    buf = LLBuffer(R, E, K, T, H, cap)
    trace = torch.full((E, R), -1, dtype=torch.int64, device="cuda")
    buf.trace_waits(trace)
    buf.set_wait_timeout_us(20_000)
    pk = buf.alloc_packed()
    buf.recv(pk)  # a fresh buffer: its count slots still hold the sentinel
    with pytest.raises(EpError):
        buf.check()
    assert (trace.cpu() >= 20_000_000).all()             # each receive waited out its 20 ms
    trace.fill_(-1)
    idx = inputs.random_topk(R, E, K, T, 0).cuda()
    x = inputs.random_x(R, T, H, 0).cuda()
    buf.dispatch(x, idx)
    buf.check()
    t = trace.cpu()
    assert (t >= 0).all() and (t < 20_000_000).all()      # every (expert, source) written, under the limit
    buf.trace_waits(None)


def test_expert_alignment_limits():
    """Alignments outside 1..65536, or whose padding would push the permuted
    row count past the int32 positions, are rejected on the host and leave
    the alignment in force unchanged."""
    ctx = Context(4, 8, 2, 16, 64, num_channels=1)
    for bad in (0, -3, 65537):
        with pytest.raises(EpError) as e:
            ctx.set_expert_alignment(bad)
        assert e.value.status == "EP_ERR_INVALID_ARG"
    assert ctx.expert_alignment == 1
    # R*T*K = 32 * 1 970 000 * 32 ~ 2.017e9: E*(alignment-1) = 2048*1023 still fits
    # below 2^31, 2048*65535 does not (the context holds a ~4 GB workspace)
    big = Context(32, 2048, 32, 1_970_000, 128, num_channels=1)
    big.set_expert_alignment(1024)
    with pytest.raises(EpError) as e:
        big.set_expert_alignment(65536)
    assert e.value.status == "EP_ERR_INVALID_ARG"
    assert big.expert_alignment == 1024
    big.close()


def test_ll_invalid_topk_is_reported_and_the_rest_exact():
    """An expert index outside [-1, E) in the low-latency send is skipped and
    flagged (EP_ERR_INVALID_INPUT at the next check); every other entry's
    slot, count and packed message equals the oracle's on the same routing
    with those entries masked."""
    import oracle as orc
    from parity_util import check_ll_microbatch_equal
    R, E, K, T, H, cap = 4, 16, 4, 10, 256, 10
    idx = inputs.random_topk(R, E, K, T, 17, 0.1)
    x = inputs.random_x(R, T, H, 17)
    bad = idx.clone()
    bad[1, 3, 2] = E
    bad[3, 9, 0] = -3
    masked = bad.clone()
    masked[1, 3, 2] = -1
    masked[3, 9, 0] = -1
    buf = LLBuffer(R, E, K, T, H, cap)
    pk = buf.dispatch(x.cuda(), bad.cuda())
    torch.cuda.synchronize()
    with pytest.raises(EpError) as e:
        buf.check()
    assert e.value.status == "EP_ERR_INVALID_INPUT"
    buf.check()  # cleared
    sent = orc.ll_send(x, masked, R, E, cap)
    o_pk = orc.ll_pack(sent, R, E, H, cap)
    check_ll_microbatch_equal(pk, sent, o_pk, R, E, T, cap)
    assert int(pk["packed_recv_count"].sum()) == int((masked >= 0).sum())
