"""FP8 rows on the normal path against the oracle: the quantised rows (codes
and scales bit-exact under round-to-nearest-even with scale = amax / 448), and
their dispatch, permute and fused dispatch (every row byte-exact)."""
import numpy as np
import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, inputs
from parity_util import bits, eq

pytestmark = pytest.mark.gpu


def _oracle_rows(x, row_q):
    """Oracle FP8 rows [R*T][row_q] (codes, scales; padding zero)."""
    xb = bits(x).reshape(-1, x.shape[-1])
    H = xb.shape[1]
    rows = np.zeros((xb.shape[0], row_q), np.uint8)
    for g in range(xb.shape[0]):
        codes, scales = orc.quantize_row(xb[g])
        rows[g, :H] = codes
        rows[g, H:H + H // 32] = scales.view(np.uint8)
    return rows


@pytest.mark.parametrize("R,E,K,T,H,C,mask_p,seed", [
    (4, 8, 2, 16, 128, 2, 0.0, 0),
    (8, 64, 8, 300, 512, 4, 0.05, 1),
    (4, 16, 4, 77, 384, 3, 0.2, 2),
])
def test_fp8_rows_dispatch_permute(R, E, K, T, H, C, mask_p, seed):
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    x = inputs.random_x(R, T, H, seed)
    if seed == 1:
        x[0, 3] = 0.0          # an all-zero token: zero scales, sign-only codes
        x[1, 5, :128] = -0.0
    w = inputs.random_weights(R, T, K, seed)
    ctx = Context(R, E, K, T, H, num_channels=C)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    lay = ctx.get_dispatch_layout(idxd)
    h = ctx.notify_dispatch(idxd, lay)
    xq = ctx.quantize_fp8(xd)
    rq = ctx.fp8_row_bytes
    n_def = H + H // 32  # defined bytes of a row (the rest is padding)
    o_rows = _oracle_rows(x, rq)
    eq(bits(xq)[:, :n_def], o_rows[:, :n_def], "fp8 rows")
    recv = ctx.dispatch_fp8(xq, idxd, wd, h)
    perm = ctx.permute_fp8(h, recv)
    fused = ctx.dispatch_permuted_fp8(xq, idxd, wd, h)
    ctx.check()
    # the oracle moves the same rows (as opaque 2-byte units)
    o_lay = orc.layout(idx, R, E)
    o_note = orc.notify(o_lay, R, E, T, C)
    rows16 = o_rows.view(np.uint16).reshape(R, T, rq // 2)
    o_disp = orc.dispatch(rows16, idx, w, o_note, R, E)
    o_perm = orc.permute(idx, o_disp["recv_x"], o_note, R, E)
    for k in ("recv_src_rank", "recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        eq(recv[k], o_disp[k], k)
    eq(bits(recv["recv_xq"])[:, :n_def], o_disp["recv_x"].view(np.uint8)[:, :n_def], "recv fp8 rows")
    eq(bits(perm["permuted_xq"])[:, :n_def], o_perm["permuted_x"].view(np.uint8)[:, :n_def], "permuted fp8 rows")
    eq(perm["perm_src_row"], o_perm["perm_src_row"], "perm_src_row")
    eq(bits(fused["permuted_xq"])[:, :n_def], o_perm["permuted_x"].view(np.uint8)[:, :n_def], "fused fp8 rows")


def test_fp8_needs_hidden_multiple_of_128():
    ctx = Context(2, 4, 2, 4, 136, num_channels=1)
    from combine_get_dispatch_histograms_gb300 import EpError
    with pytest.raises(EpError):
        ctx.quantize_fp8(torch.zeros(2, 4, 136, dtype=torch.bfloat16, device="cuda"))
