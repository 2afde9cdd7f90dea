"""Guard bands around every output: each output tensor is a slice in the
middle of a larger allocation whose head and tail are filled with a canary
pattern; after the kernels the canaries must be untouched (no write outside
an output's bounds).  Covers the normal path (layout, notify, dispatch,
permute, fused dispatch, FP8 rows, one-pass FP8 dispatches, hierarchical
staging, combine) and the low-latency path (receive outputs, combine)."""
import pytest
import torch

from combine_get_dispatch_histograms_gb300 import Context, LLBuffer, inputs

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
CANARY = 0xA5


class Guarded:
    def __init__(self):
        self.bufs = []

    def empty(self, *shape, dtype):
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty(0, dtype=dtype).element_size()
        raw = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.bufs.append((raw, nbytes))
        return raw[GUARD:GUARD + nbytes].view(dtype).view(*shape)

    def check(self):
        torch.cuda.synchronize()
        for raw, nbytes in self.bufs:
            head, tail = raw[:GUARD], raw[GUARD + nbytes:]
            assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), "write outside an output"


@pytest.mark.parametrize("N", [1, 2])
def test_normal_path_stays_in_bounds(N):
    R, E, K, T, H, C = 8, 64, 8, 300, 256, 4
    idx = inputs.random_topk(R, E, K, T, 70, 0.1).cuda()
    x = inputs.random_x(R, T, H, 70).cuda()
    w = inputs.random_weights(R, T, K, 70).cuda()
    ctx = Context(R, E, K, T, H, num_channels=C, num_nodes=N)
    g = Guarded()
    i32 = lambda *s: g.empty(*s, dtype=torch.int32)
    lay = dict(num_tokens_per_expert=i32(R, E), num_tokens_per_rank=i32(R, R),
               is_token_in_rank=g.empty(R, T, R, dtype=torch.uint8))
    if N > 1:
        lay["num_tokens_per_node"] = i32(R, N)
        lay["is_token_in_node"] = g.empty(R, T, N, dtype=torch.uint8)
    ctx.get_dispatch_layout(idx, out=lay)
    L = E // R
    from combine_get_dispatch_histograms_gb300 import Handle
    h = Handle(recv_count=i32(R, R), recv_offsets=i32(R, R), num_recv_tokens=i32(R), rank_base=i32(R + 1),
               num_recv_per_expert=i32(R, L), expert_offsets=i32(R, L), perm_rank_base=i32(R + 1),
               channel_prefix_matrix=i32(R, R, C), send_pos=i32(R, T, R), perm_pos=i32(R, T, K))
    if N > 1:
        h["stage_base"] = i32(R + 1)
        h["stage_pos"] = i32(R, T, N)
    h = ctx.notify_dispatch(idx, lay, handle=h)
    nr, npm, ns = h.num_recv_rows, h.num_perm_rows, h.num_stage_rows
    recv = dict(recv_x=g.empty(nr, H, dtype=torch.bfloat16), recv_src_rank=i32(nr), recv_src_idx=i32(nr),
                recv_topk_idx=i32(nr, K), recv_topk_weights=g.empty(nr, K, dtype=torch.float32))
    if N > 1:
        st = dict(staging=g.empty(ns, H, dtype=torch.bfloat16), stage_src_rank=i32(ns), stage_src_idx=i32(ns))
        ctx.dispatch_hier(x, idx, w, h, out=recv, staging=st)
    else:
        ctx.dispatch(x, idx, w, h, out=recv)
    perm = dict(permuted_x=g.empty(npm, H, dtype=torch.bfloat16), perm_src_row=i32(npm))
    ctx.permute(h, recv, out=perm)
    fused = dict(permuted_x=g.empty(npm, H, dtype=torch.bfloat16), perm_src_token=i32(npm),
                 perm_weight=g.empty(npm, dtype=torch.float32))
    ctx.dispatch_permuted(x, idx, w, h, out=fused)
    rq = ctx.fp8_row_bytes
    xq = g.empty(R * T, rq, dtype=torch.uint8)
    ctx.quantize_fp8(x, out=xq)
    ctx.dispatch_permuted_fp8(xq, idx, w, h, out=dict(permuted_xq=g.empty(npm, rq, dtype=torch.uint8),
                                                      perm_src_token=i32(npm),
                                                      perm_weight=g.empty(npm, dtype=torch.float32)))
    ctx.dispatch_permuted_quant(x, idx, w, h, out=dict(permuted_xq=g.empty(npm, rq, dtype=torch.uint8),
                                                       perm_src_token=i32(npm),
                                                       perm_weight=g.empty(npm, dtype=torch.float32)))
    ctx.dispatch_quant(x, idx, w, h, out=dict(recv_xq=g.empty(nr, rq, dtype=torch.uint8), recv_src_rank=i32(nr),
                                              recv_src_idx=i32(nr), recv_topk_idx=i32(nr, K),
                                              recv_topk_weights=g.empty(nr, K, dtype=torch.float32)))
    out = g.empty(R, T, H, dtype=torch.bfloat16)
    ctx.combine(h, perm["permuted_x"], idx, w, out=out, hier=N > 1)
    ctx.check()
    g.check()


def test_low_latency_stays_in_bounds():
    R, E, K, T, H, cap = 8, 32, 4, 40, 256, 20
    idx = inputs.random_topk(R, E, K, T, 71, 0.05).cuda()
    x = inputs.random_x(R, T, H, 71).cuda()
    w = inputs.random_weights(R, T, K, 71).cuda()
    buf = LLBuffer(R, E, K, T, H, cap)
    g = Guarded()
    L = E // R
    pk = dict(packed_x=g.empty(R, L, R * cap, H, dtype=torch.uint8),
              packed_scales=g.empty(R, L, R * cap, H // 128, dtype=torch.float32),
              packed_src_info=g.empty(R, L, R * cap, 2, dtype=torch.int32),
              packed_recv_count=g.empty(R, L, dtype=torch.int32), layout_range=g.empty(R, L, R, 2, dtype=torch.int32),
              slot=g.empty(R, T, K, dtype=torch.int32))
    out = g.empty(R, T, H, dtype=torch.bfloat16)
    out.zero_()
    y = torch.randn(R, L, R * cap, H, device="cuda").to(torch.bfloat16)
    for t0 in range(0, T, cap):
        buf.dispatch(x, idx, t0, min(cap, T - t0), out=pk)
        buf.combine(y, idx, w, pk, t0, min(cap, T - t0), out=out)
    buf.check()
    g.check()
