"""The fused layout + notify (two launches instead of three) against the
oracle: every layout output and every handle array, bit for bit, flat and
hierarchical, with and without the host wait, repeated on one context (the
completion counters re-arm), and inside a captured CUDA graph."""
import numpy as np
import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, EpError, inputs
from parity_util import eq

pytestmark = pytest.mark.gpu

HANDLE = ("recv_count", "num_recv_tokens", "recv_offsets", "rank_base", "num_recv_per_expert",
          "expert_offsets", "perm_rank_base", "channel_prefix_matrix", "send_pos")


def _check(ctx, idx, lay, h, N):
    R, E, T, C = ctx.R, ctx.E, ctx.T, ctx.C
    o_lay = orc.layout(idx, R, E, num_nodes=N if N > 1 else 0)
    for k in o_lay:
        eq(lay[k], o_lay[k], k)
    o_note = orc.notify(o_lay, R, E, T, C)
    for k in HANDLE:
        eq(h[k], o_note[k], k)
    o_disp = orc.dispatch(np.zeros((R, T, 8), np.uint16), idx, inputs.random_weights(R, T, ctx.K, 0), o_note, R, E)
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    eq(h["perm_pos"], o_perm["perm_pos"], "perm_pos")
    if N > 1:
        sb, sp = orc.hier_stage_pos(o_lay, R, T, N)
        eq(h["stage_base"], sb, "stage_base")
        eq(h["stage_pos"], sp, "stage_pos")
    return o_note


@pytest.mark.parametrize("R,E,K,T,C,N,mask_p,seed", [
    (4, 8, 2, 600, 3, 1, 0.1, 1),
    (8, 256, 8, 700, 8, 1, 0.0, 2),
    (16, 4096, 8, 96, 4, 1, 0.0, 3),
    (64, 128, 32, 40, 8, 1, 0.05, 4),
    (8, 32, 4, 300, 4, 2, 0.05, 5),     # hierarchical
    (32, 256, 8, 120, 8, 4, 0.05, 6),   # hierarchical, 4 nodes
    (4, 8, 2, 0, 2, 1, 0.0, 7),         # no tokens
    (4, 8, 2, 100, 2, 1, 1.0, 8),       # everything masked
])
def test_layout_notify(R, E, K, T, C, N, mask_p, seed):
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    ctx = Context(R, E, K, T, 64, num_channels=C, num_nodes=N)
    idxd = idx.cuda()
    for rep in range(2):  # the counters re-arm
        lay, h = ctx.layout_notify(idxd)
        ctx.check()
        o_note = _check(ctx, idx, lay, h, N)
        assert h.num_recv_rows == int(o_note["rank_base"][R])
        assert h.num_perm_rows == int(o_note["perm_rank_base"][R])
        assert list(h.host_num_recv_tokens) == list(o_note["num_recv_tokens"])
    # the same handle as the separate calls
    lay2 = ctx.get_dispatch_layout(idxd, nodes=N > 1)
    h2 = ctx.notify_dispatch(idxd, lay2)
    for k in h:
        assert torch.equal(h[k], h2[k]), k
    for k in lay:
        assert torch.equal(lay[k], lay2[k]), k


def test_layout_notify_no_wait_in_a_graph():
    R, E, K, T, C = 8, 64, 4, 300, 4
    ctx = Context(R, E, K, T, 64, num_channels=C)
    idxd = torch.empty(R, T, K, dtype=torch.int64, device="cuda")
    idxd.copy_(inputs.random_topk(R, E, K, T, 20, 0.05))
    lay, h = ctx.layout_notify(idxd, wait=False)  # eager once, outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ctx.layout_notify(idxd, handle=h, out=lay, wait=False)
    for seed in (21, 22):
        idx = inputs.random_topk(R, E, K, T, seed, 0.05)
        idxd.copy_(idx)
        g.replay()
        torch.cuda.synchronize()
        ctx.check()
        _check(ctx, idx, lay, h, 1)


def test_layout_notify_invalid_topk():
    R, E, K, T = 4, 8, 2, 20
    idx = inputs.random_topk(R, E, K, T, 30)
    idx[1, 3, 0] = E
    ctx = Context(R, E, K, T, 64, num_channels=2)
    with pytest.raises(EpError) as e:
        ctx.layout_notify(idx.cuda())
    assert e.value.status == "EP_ERR_INVALID_INPUT"
    with pytest.raises(EpError):
        ctx.check()
