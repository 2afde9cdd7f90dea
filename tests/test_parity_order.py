"""GPU combine kernels on inputs built so that the fp32 summation order shows
through the bf16 output (exact cancellations, an fma-only residual), against
the oracle, bit-exactly: rank order and fused multiply-adds of the flat
combine, the node grouping of the hierarchical combine, and the k order of the
low-latency combine.  Random data cannot catch an order mistake: bf16 rounding
hides fp32-level differences."""
import numpy as np
import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, LLBuffer
from parity_util import eq

pytestmark = pytest.mark.gpu

R, E, K, H, N = 4, 8, 4, 64, 2
BIG = float(2 ** 25)
W0 = float(np.float32(1.0 + 2.0 ** -23))
# (experts of token 0, weights, x value): the cases of tests/test_oracle_order.py,
# plus the same rows in permuted k order, one token each
CASES = [
    ([0, 2, 4, -1], [BIG, -BIG, 1.0, 0.0], 1.0),     # rank order: 1
    ([0, 2, 4, -1], [1.0, BIG, -BIG, 0.0], 1.0),     # rank order: 0
    ([0, 1, -1, -1], [W0, -W0, 0.0, 0.0], 1.5),      # fma residual on one rank
    ([0, 4, 6, -1], [BIG, -BIG, 1.0, 0.0], 1.0),     # node grouping: flat 1, hierarchical 0
    ([4, 0, 2, -1], [BIG, -BIG, 1.0, 0.0], 1.0),     # k order differs from rank order
    ([6, 4, 0, 2], [1.0, BIG, -BIG, 3.0], 1.0),
]


def _inputs():
    T = len(CASES)
    idx = np.full((R, T, K), -1, np.int64)
    w = np.zeros((R, T, K), np.float32)
    x = np.zeros((R, T, H), np.float32)
    for t, (ex, ws, xv) in enumerate(CASES):
        idx[0, t] = ex
        w[0, t] = ws
        x[0, t] = xv
    return T, torch.from_numpy(idx), torch.from_numpy(w), torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("hier", [False, True], ids=["flat", "hierarchical"])
def test_combine_order_cases(hier):
    T, idx, w, x = _inputs()
    ctx = Context(R, E, K, T, H, num_channels=1, num_nodes=N)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    lay = ctx.get_dispatch_layout(idxd)
    h = ctx.notify_dispatch(idxd, lay)
    recv = ctx.dispatch(xd, idxd, wd, h)
    perm = ctx.permute(h, recv)
    out = ctx.combine(h, perm["permuted_x"], idxd, wd, hier=hier)
    ctx.check()
    o = orc.run_normal(x, idx, w, R, E, 1)
    if hier:
        exp = orc.combine_hier(o["permute"]["permuted_x"], o["permute"]["perm_pos"], idx, w, R, E, N)
    else:
        exp = o["out"]
    eq(out, exp, "combine order cases")
    # the cases really separate the orders: flat and hierarchical differ on the grouping case
    flat = o["out"][0, 3, 0]
    hr = orc.combine_hier(o["permute"]["permuted_x"], o["permute"]["perm_pos"], idx, w, R, E, N)[0, 3, 0]
    assert flat != hr


def test_ll_combine_k_order_cases():
    T, idx, w, x = _inputs()
    cap = T
    buf = LLBuffer(R, E, K, T, 128, cap)
    x128 = x[..., :1].expand(R, T, 128).contiguous()
    xd, idxd, wd = x128.cuda(), idx.cuda(), w.cuda()
    pk = buf.dispatch(xd, idxd)
    sent = orc.ll_send(x128, idx, R, E, cap)
    o_pk = orc.ll_pack(sent, R, E, 128, cap)
    y = orc.ll_dequant(o_pk["packed_x"], o_pk["packed_scales"])
    out = buf.combine(torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda(), idxd, wd, pk)
    buf.check()
    exp = orc.ll_combine(y, idx, w, sent["slot"], o_pk["layout_range"], R, E, cap)
    eq(out, exp, "ll combine order cases")
    # the k order shows: [1, 2^25, -2^25] sums to 0 and [2^25, -2^25, 1] to 1,
    # whatever ranks the experts sit on
    assert exp[0, 1, 0] != exp[0, 4, 0]
