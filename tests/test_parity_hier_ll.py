"""GPU vs oracle for the hierarchical staging and the low-latency (FP8) path."""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import LLBuffer, inputs
from parity_util import compare_normal, eq, run_gpu_ll, bits

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# hierarchical (node, then rank) staging
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("R,N,E,K,T,H,C,mask_p,seed", [
    (8, 2, 32, 4, 300, 64, 4, 0.0, 1),
    (32, 4, 256, 8, 120, 128, 8, 0.05, 2),
    (8, 8, 16, 2, 77, 64, 2, 0.2, 3),     # one rank per node
    (4, 1 + 1, 8, 2, 0, 64, 2, 0.0, 4),   # no tokens
])
@pytest.mark.parametrize("hier", [True, False], ids=["staged", "flat"])
def test_hier_and_flat_with_nodes(R, N, E, K, T, H, C, mask_p, seed, hier):
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    compare_normal(R, E, K, T, H, C, x, idx, w, nodes=N, hier=hier)


def test_hier_workload_shape_small():
    w = inputs.WORKLOADS["hier"].replace(T=64, H=256)
    x, idx, wts = inputs.make_inputs(w, seed=0)
    compare_normal(w.R, w.E, w.K, w.T, w.H, w.num_channels, x, idx, wts, nodes=w.num_nodes, hier=True)


# ---------------------------------------------------------------------------
# low-latency mode
# ---------------------------------------------------------------------------

def _cudart():
    for cand in ("/usr/local/cuda/lib64/libcudart.so", ctypes.util.find_library("cudart")):
        if cand and os.path.exists(cand):
            lib = ctypes.CDLL(cand)
            lib.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
            return lib
    pytest.skip("libcudart not found for the count-slot read-back")


def read_counts(buf, which):
    lib = _cudart()
    n = buf.E * buf.R
    host = np.empty((buf.E, buf.R), np.int32)
    torch.cuda.synchronize()
    rc = lib.cudaMemcpy(host.ctypes.data, buf.count_slots(which), n * 4, 2)  # device -> host
    assert rc == 0
    return host


def check_ll_microbatch(pk, sent, o_pk, R, E, K, T, H, cap, t0, n, idx):
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


@pytest.mark.parametrize("R,E,K,T,H,cap,mbs,mask_p,seed", [
    (4, 8, 2, 16, 128, 16, [(0, 16)], 0.0, 0),
    (16, 256, 8, 40, 512, 40, [(0, 40)], 0.0, 1),
    (8, 64, 8, 50, 256, 20, [(0, 20), (20, 20), (40, 10)], 0.05, 2),   # microbatches, ragged tail
    (2, 4, 2, 9, 384, 9, [(0, 9)], 0.3, 3),
    (4, 8, 2, 6, 128, 6, [(0, 0)], 0.0, 4),                             # empty microbatch
    (1, 1, 1, 5, 128, 5, [(0, 5)], 0.0, 5),                             # one rank, one expert
    (64, 64, 8, 4, 128, 4, [(0, 4)], 0.0, 6),                           # 64 ranks, one expert per rank
    (4, 16, 16, 8, 16384, 8, [(0, 8)], 0.1, 7),                         # largest hidden, K = 16
    (4, 8, 2, 3, 256, 1, [(0, 1), (1, 1), (2, 1)], 0.0, 8),             # cap 1: one token per microbatch
    (2, 64, 32, 6, 256, 6, [(0, 6)], 0.0, 9),                           # K = 32
])
def test_low_latency(R, E, K, T, H, cap, mbs, mask_p, seed):
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    x = inputs.random_x(R, T, H, seed)
    w = inputs.random_weights(R, T, K, seed)
    from combine_get_dispatch_histograms_gb300 import LLBuffer
    buf = LLBuffer(R, E, K, T, H, cap)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    out = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
    o_out = np.zeros((R, T, H), np.uint16)
    out_r = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
    o_out_r = np.zeros((R, T, H), np.uint16)
    for t0, n in mbs:
        pk = buf.send(xd, idxd, t0, n)
        counts = read_counts(buf, buf.current_buffer)
        sent = orc.ll_send(x, idx, R, E, cap, t0, n)
        # every count slot written after the send, none left at the sentinel
        eq(counts, sent["counts"], "count slots")
        assert counts.sum() == (idx.numpy()[:, t0:t0 + n] >= 0).sum()
        buf.recv(pk)
        torch.cuda.synchronize()
        o_pk = orc.ll_pack(sent, R, E, H, cap)
        check_ll_microbatch(pk, sent, o_pk, R, E, K, T, H, cap, t0, n, idx)
        # identity expert on the oracle's packed rows, then the BF16 combine
        y = orc.ll_dequant(o_pk["packed_x"], o_pk["packed_scales"])
        yd = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda()
        buf.combine(yd, idxd, wd, pk, t0, n, out=out)
        orc.ll_combine(y, idx, w, sent["slot"], o_pk["layout_range"], R, E, cap, t0, n, out=o_out)
        # an expert output with a different row in every packed slot
        L = E // R
        yr = inputs.random_rows(R * L * R * cap, H, seed=seed * 17 + t0).view(R, L, R * cap, H)
        buf.combine(yr.cuda(), idxd, wd, pk, t0, n, out=out_r)
        orc.ll_combine(yr, idx, w, sent["slot"], o_pk["layout_range"], R, E, cap, t0, n, out=o_out_r)
    buf.check()
    torch.cuda.synchronize()
    eq(out, o_out, "ll combine")
    eq(out_r, o_out_r, "ll combine of distinct expert rows")


def test_low_latency_ping_pong_resets_counts():
    R, E, K, T, H, cap = 4, 8, 2, 12, 128, 12
    idx = inputs.random_topk(R, E, K, T, 5)
    x = inputs.random_x(R, T, H, 5)
    from combine_get_dispatch_histograms_gb300 import LLBuffer
    buf = LLBuffer(R, E, K, T, H, cap)
    assert (read_counts(buf, 0) == -1).all() and (read_counts(buf, 1) == -1).all()
    pk = buf.dispatch(x.cuda(), idx.cuda())
    assert buf.current_buffer == 0
    assert (read_counts(buf, 0) >= 0).all() and (read_counts(buf, 1) == -1).all()
    pk2 = buf.dispatch(x.cuda(), idx.cuda())
    assert buf.current_buffer == 1
    # the second send re-armed buffer 0 to the sentinel and published buffer 1
    assert (read_counts(buf, 0) == -1).all() and (read_counts(buf, 1) >= 0).all()
    buf.check()
    for k in ("packed_recv_count", "layout_range", "slot"):
        assert torch.equal(pk[k], pk2[k])


def test_low_latency_workload_shapes_small():
    for name in ("decode", "skewed"):
        wl = inputs.WORKLOADS[name].replace(T=48, H=256, ll_cap=16)
        x, idx, w = inputs.make_inputs(wl, seed=0)
        R, E, K, T, H, cap = wl.R, wl.E, wl.K, wl.T, wl.H, wl.ll_cap
        mbs = [(t0, min(cap, T - t0)) for t0 in range(0, T, cap)]
        buf, outs = run_gpu_ll(R, E, K, T, H, cap, x, idx, mbs)
        for (t0, n), pk in zip(mbs, outs):
            sent = orc.ll_send(x, idx, R, E, cap, t0, n)
            o_pk = orc.ll_pack(sent, R, E, H, cap)
            check_ll_microbatch(pk, sent, o_pk, R, E, K, T, H, cap, t0, n, idx)


def test_low_latency_layer_in_cuda_graph():
    """The low-latency layer (send, receive, combine) has static shapes and no
    host synchronisation: captured once in a CUDA graph, each replay gives the
    eager result."""
    R, E, K, T, H, cap = 8, 64, 4, 24, 256, 24
    idx = inputs.random_topk(R, E, K, T, 21, 0.1)
    x = inputs.random_x(R, T, H, 21)
    w = inputs.random_weights(R, T, K, 21)
    from combine_get_dispatch_histograms_gb300 import LLBuffer
    buf = LLBuffer(R, E, K, T, H, cap)
    xd, idxd, wd = x.cuda(), idx.cuda(), w.cuda()
    sent = orc.ll_send(x, idx, R, E, cap)
    o_pk = orc.ll_pack(sent, R, E, H, cap)
    y = orc.ll_dequant(o_pk["packed_x"], o_pk["packed_scales"])
    yd = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda()
    o_out = orc.ll_combine(y, idx, w, sent["slot"], o_pk["layout_range"], R, E, cap)
    pk = buf.alloc_packed()
    out = torch.zeros(R, T, H, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        buf.dispatch(xd, idxd, out=pk)
        buf.combine(yd, idxd, wd, pk, out=out)
    s.synchronize()
    eq(out, o_out, "eager")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        buf.dispatch(xd, idxd, out=pk)
        buf.combine(yd, idxd, wd, pk, out=out)
    for _ in range(3):
        out.zero_()
        pk["packed_recv_count"].fill_(-5)
        g.replay()
        torch.cuda.synchronize()
        buf.check()
        eq(out, o_out, "graph replay")
        eq(pk["packed_recv_count"], o_pk["packed_recv_count"], "graph replay counts")


def test_two_microbatches_on_two_streams():
    """Dual-microbatch overlap ([P1] 高吞吐量模式, dual-batch overlap): two
    low-latency buffers, each sending, receiving and combining its own
    microbatch on its own stream at the same time (nothing waits across the
    streams).  Each stream's packed rows, counts and combine output (of an
    expert output with a distinct row per packed slot) equal the oracle's."""
    R, E, K, T, H, cap = 8, 64, 8, 96, 256, 96
    L = E // R
    bufs = [LLBuffer(R, E, K, T, H, cap) for _ in range(2)]
    ins, ys = [], []
    for seed in (31, 32):
        idx = inputs.random_topk(R, E, K, T, seed, 0.05)
        ins.append((inputs.random_x(R, T, H, seed), idx, inputs.random_weights(R, T, K, seed)))
        ys.append(inputs.random_rows(R * L * R * cap, H, seed=seed).view(R, L, R * cap, H))
    dev = [(x.cuda(), idx.cuda(), w.cuda(), y.cuda()) for (x, idx, w), y in zip(ins, ys)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    main = torch.cuda.current_stream()
    res = []
    for st, b, (x, idx, w, y) in zip(streams, bufs, dev):
        st.wait_stream(main)
        with torch.cuda.stream(st):
            pk = b.dispatch(x, idx)
            out = b.combine(y, idx, w, pk)
        res.append((pk, out))
    for st in streams:
        main.wait_stream(st)
    torch.cuda.synchronize()
    for b, (pk, out), (x, idx, w), y in zip(bufs, res, ins, ys):
        b.check()
        sent = orc.ll_send(x, idx, R, E, cap)
        o_pk = orc.ll_pack(sent, R, E, H, cap)
        check_ll_microbatch(pk, sent, o_pk, R, E, K, T, H, cap, 0, T, idx)
        o_out = orc.ll_combine(y, idx, w, sent["slot"], o_pk["layout_range"], R, E, cap)
        eq(out, o_out, "combine of the overlapped microbatch")


def test_low_latency_x_only_16_byte_aligned():
    """x may be only 16-byte aligned (the documented requirement): the send
    then loads each lane's channels with two 16-byte loads instead of one
    32-byte load; the messages and the combine equal the oracle's."""
    R, E, K, T, H, cap = 8, 64, 8, 20, 1024, 20
    idx = inputs.random_topk(R, E, K, T, 41, 0.1)
    x = inputs.random_x(R, T, H, 41)
    w = inputs.random_weights(R, T, K, 41)
    big = torch.empty(R * T * H + 8, dtype=torch.bfloat16, device="cuda")
    xd = big[8:].view(R, T, H)          # 16 bytes past a 32-byte boundary
    assert xd.data_ptr() % 32 == 16
    xd.copy_(x.cuda())
    buf = LLBuffer(R, E, K, T, H, cap)
    pk = buf.dispatch(xd, idx.cuda())
    L = E // R
    yr = inputs.random_rows(R * L * R * cap, H, seed=41).view(R, L, R * cap, H)
    out = buf.combine(yr.cuda(), idx.cuda(), w.cuda(), pk)
    torch.cuda.synchronize()
    buf.check()
    sent = orc.ll_send(x, idx, R, E, cap)
    o_pk = orc.ll_pack(sent, R, E, H, cap)
    check_ll_microbatch(pk, sent, o_pk, R, E, K, T, H, cap, 0, T, idx)
    eq(out, orc.ll_combine(yr, idx, w, sent["slot"], o_pk["layout_range"], R, E, cap), "ll combine")
