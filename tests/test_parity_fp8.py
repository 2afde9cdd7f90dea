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


def _bf16_values_up_to(a_bits: int) -> np.ndarray:
    """Every finite bf16 value v with |v| <= the bf16 value a, both signs (bit patterns)."""
    pos = np.arange(0, 0x7f80, dtype=np.uint32)
    mag = (pos << 16).view(np.float32)
    a = np.array([a_bits << 16], np.uint32).view(np.float32)[0]
    keep = pos[mag <= a].astype(np.uint16)
    return np.concatenate([keep, keep | np.uint16(0x8000)])


def test_quantize_every_bf16_value_for_many_scales():
    """Exhaustive over x: for each block maximum a (so scale = a / 448), every
    bf16 value with |x| <= a, in blocks of 128 led by a; codes and scales
    bit-exact against the oracle, on the normal-mode quantiser and on the
    low-latency send (both use the same codec)."""
    rng = np.random.default_rng(5)
    special = [0x43e0, 0x4360, 0x4460,  # 448, 224, 896: scales 1, 1/2, 2 (exact quotients, e4m3 ties)
               0x3f80, 0x4040, 0x4030, 0x3e99, 0x3a83, 0x3c8c, 0x40a0, 0x40e0, 0x449a,
               0x7f7f,  # largest finite bf16
               0x0080,  # smallest normal bf16
               0x0001, 0x0040,  # subnormal block maxima
               0x11DF, 0x11E0, 0x11E1]  # scales on both sides of 2^-100 (the division fallback)
    amaxes = (special + [int(b) for b in rng.integers(0x2000, 0x5000, size=10)]
              + [int(b) for b in rng.integers(0x0001, 0x7F80, size=16)])
    blocks = []
    for a in amaxes:
        vals = _bf16_values_up_to(a)
        vals = vals[np.argsort(rng.random(len(vals)))]
        nb = -(-len(vals) // 127)
        pad = np.zeros(nb * 127, np.uint16)
        pad[:len(vals)] = vals
        blk = np.concatenate([np.full((nb, 1), a, np.uint16), pad.reshape(nb, 127)], axis=1)
        blocks.append(blk)
    blocks = np.concatenate(blocks)
    H = 128 * 64
    T = -(-blocks.shape[0] // 64)
    allb = np.zeros((T * 64, 128), np.uint16)
    allb[:blocks.shape[0]] = blocks
    xb = allb.reshape(T, H)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).reshape(1, T, H)
    o_rows = np.stack([np.concatenate([c, s.view(np.uint8)]) for c, s in map(orc.quantize_row, xb)])
    n_def = H + H // 32
    # normal-mode quantiser
    ctx = Context(1, 1, 1, T, H, num_channels=1)
    xq = ctx.quantize_fp8(x.cuda())
    ctx.check()
    eq(bits(xq)[:, :n_def], o_rows, "fp8 rows (exhaustive bf16 x)")
    # low-latency send: one rank, one expert, every token sent once (slot = t)
    from combine_get_dispatch_histograms_gb300 import LLBuffer
    buf = LLBuffer(1, 1, 1, T, H, T)
    pk = buf.dispatch(x.cuda(), torch.zeros(1, T, 1, dtype=torch.int64, device="cuda"))
    buf.check()
    eq(pk["packed_x"][0, 0, :T], o_rows[:, :H], "LL message codes (exhaustive bf16 x)")
    eq(pk["packed_scales"][0, 0, :T], o_rows[:, H:].view(np.float32), "LL message scales")


@pytest.mark.parametrize("R,E,K,T,H,C,mask_p,align,seed,wait", [
    (4, 8, 2, 16, 128, 2, 0.0, 1, 0, True),
    (8, 64, 8, 300, 512, 4, 0.05, 1, 1, True),
    (4, 16, 4, 77, 384, 3, 0.2, 1, 2, True),
    (8, 256, 8, 200, 7168, 8, 0.0, 1, 3, True),      # the prefill row size
    (4, 16, 4, 150, 256, 4, 0.1, 16, 4, True),       # expert-aligned blocks
    (4, 16, 4, 150, 256, 4, 0.1, 1, 5, False),       # no-wait notify, worst-case buffers
    (4, 8, 2, 0, 128, 2, 0.0, 1, 6, True),           # no tokens
    (4, 16, 4, 40, 16384, 2, 0.0, 1, 7, True),       # largest hidden: two staged rows per CTA
])
def test_quantise_and_dispatch_in_one_pass(R, E, K, T, H, C, mask_p, align, seed, wait):
    """ep_dispatch_permuted_quant gives the bytes of quantize_fp8 followed by
    dispatch_permuted_fp8, and the oracle's FP8 rows in the oracle's order."""
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    x = inputs.random_x(R, T, H, seed)
    if seed == 1:
        x[0, 3] = 0.0
    w = inputs.random_weights(R, T, K, seed)
    ctx = Context(R, E, K, T, H, num_channels=C, expert_alignment=align)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    lay = ctx.get_dispatch_layout(idxd)
    h = ctx.notify_dispatch(idxd, lay, wait=wait)
    one = ctx.dispatch_permuted_quant(xd, idxd, wd, h)
    ctx.check()
    rq = ctx.fp8_row_bytes
    n_def = H + H // 32
    o_note = orc.notify(orc.layout(idx, R, E), R, E, T, C, align=align)
    P = int(o_note["perm_rank_base"][R])
    o_rows = _oracle_rows(x, rq)
    pp = h["perm_pos"].cpu().numpy()
    eq(pp, orc.permute(idx, np.zeros((int(o_note["rank_base"][R]), 8), np.uint16), o_note, R, E)["perm_pos"],
       "perm_pos")
    got = bits(one["permuted_xq"])[:P]
    tok = bits(one["perm_src_token"])[:P]
    wgt = bits(one["perm_weight"])[:P]
    wn = w.numpy()
    for s_, t_, k_ in zip(*np.nonzero(pp >= 0)):
        r = pp[s_, t_, k_]
        assert tok[r] == s_ * T + t_
        assert wgt[r] == wn[s_, t_, k_]
        eq(got[r, :n_def], o_rows[s_ * T + t_, :n_def], f"row {r}")
    if T > 0 and wait:
        # byte for byte the two-pass form
        xq = ctx.quantize_fp8(xd)
        two = ctx.dispatch_permuted_fp8(xq, idxd, wd, h)
        ctx.check()
        used = np.zeros(P, bool)
        used[pp[pp >= 0]] = True
        eq(got[used][:, :n_def], bits(two["permuted_xq"])[:P][used][:, :n_def], "one pass vs two passes")
        eq(tok[used], bits(two["perm_src_token"])[:P][used], "perm_src_token")


@pytest.mark.parametrize("R,E,K,T,H,C,mask_p,seed,wait", [
    (4, 8, 2, 16, 128, 2, 0.0, 0, True),
    (8, 64, 8, 300, 512, 4, 0.05, 1, True),
    (16, 256, 8, 100, 7168, 8, 0.1, 2, True),
    (4, 16, 4, 150, 256, 4, 0.1, 3, False),        # no-wait notify, worst-case buffers
    (4, 8, 2, 0, 128, 2, 0.0, 4, True),            # no tokens
    (4, 16, 4, 40, 16384, 2, 0.0, 5, True),        # largest hidden
])
def test_quantise_and_scatter_in_one_pass(R, E, K, T, H, C, mask_p, seed, wait):
    """ep_dispatch_quant: the receive layout of quantize_fp8 + dispatch_fp8, and
    the oracle's metadata and FP8 rows."""
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    ctx = Context(R, E, K, T, H, num_channels=C)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    h = ctx.notify_dispatch(idxd, ctx.get_dispatch_layout(idxd), wait=wait)
    one = ctx.dispatch_quant(xd, idxd, wd, h, out=None if wait else ctx_recv_fp8(ctx))
    ctx.check()
    rq = ctx.fp8_row_bytes
    n_def = H + H // 32
    o_note = orc.notify(orc.layout(idx, R, E), R, E, T, C)
    nr = int(o_note["rank_base"][R])
    o_rows = _oracle_rows(x, rq)
    rows16 = o_rows.view(np.uint16).reshape(R, T, rq // 2) if T > 0 else np.zeros((R, 0, rq // 2), np.uint16)
    o_disp = orc.dispatch(rows16, idx, w, o_note, R, E)
    for k in ("recv_src_rank", "recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        eq(bits(one[k])[:nr], o_disp[k], k)
    eq(bits(one["recv_xq"])[:nr, :n_def], o_disp["recv_x"].view(np.uint8)[:, :n_def], "recv FP8 rows")


def ctx_recv_fp8(ctx):
    rows = ctx.max_rows[0]
    return dict(recv_xq=torch.empty(rows, ctx.fp8_row_bytes, dtype=torch.uint8, device="cuda"),
                recv_src_rank=torch.empty(rows, dtype=torch.int32, device="cuda"),
                recv_src_idx=torch.empty(rows, dtype=torch.int32, device="cuda"),
                recv_topk_idx=torch.empty(rows, ctx.K, dtype=torch.int32, device="cuda"),
                recv_topk_weights=torch.empty(rows, ctx.K, dtype=torch.float32, device="cuda"))
