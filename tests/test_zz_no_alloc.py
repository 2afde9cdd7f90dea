"""The allocation-free layout entry point, called through the C ABI.

This entry point serves callers that may not allocate device memory
themselves (for example a plug-in whose host runtime owns all of HBM through
its own pool): it keeps its scratch in a fixed array inside the library.
Its outputs are compared with the oracle's layout and with the context-based
ep_get_dispatch_layout on the same inputs, on two calls in a row; an
out-of-range expert index must come back as bit 1 of status_out, and a call
without status_out must still give the same outputs.
The file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

import oracle as orc
from combine_get_dispatch_histograms_gb300 import Context, _lib, inputs
from parity_util import eq

pytestmark = pytest.mark.gpu

KEYS = ("num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank")
NODE_KEYS = ("num_tokens_per_node", "is_token_in_node")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, R, E, K, T, N, idx, with_nodes, with_status=True):
    dev = idx.device
    o = dict(
        num_tokens_per_expert=torch.full((R, E), -7, dtype=torch.int32, device=dev),
        num_tokens_per_rank=torch.full((R, R), -7, dtype=torch.int32, device=dev),
        is_token_in_rank=torch.full((R, T, R), 9, dtype=torch.uint8, device=dev),
    )
    if with_nodes:
        o["num_tokens_per_node"] = torch.full((R, N), -7, dtype=torch.int32, device=dev)
        o["is_token_in_node"] = torch.full((R, T, N), 9, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev) if with_status else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.ep_get_dispatch_layout_noalloc(
        R, E, K, T, N, _p(idx), _p(o["num_tokens_per_expert"]), _p(o["num_tokens_per_rank"]),
        _p(o["is_token_in_rank"]), _p(o.get("num_tokens_per_node")), _p(o.get("is_token_in_node")),
        _p(status), stream)
    assert rc == 0, lib.ep_last_error()
    torch.cuda.synchronize()
    return o, (int(status.item()) if with_status else None)


@pytest.mark.parametrize("R,E,K,T,N,mask_p,seed", [
    (4, 8, 2, 16, 1, 0.0, 0),        # the tiny worked shape
    (8, 256, 8, 4096, 1, 0.0, 1),    # the prefill routing
    (32, 256, 8, 700, 4, 0.05, 2),   # nodes, masks, ragged last tile
    (4, 8, 2, 0, 2, 0.0, 3),         # no tokens
])
def test_noalloc_layout_equals_oracle_and_context_layout_twice(R, E, K, T, N, mask_p, seed):
    lib = _lib.load()
    idx = inputs.random_topk(R, E, K, T, seed, mask_p)
    idxd = idx.cuda()
    with_nodes = N > 1
    exp = orc.layout(idx, R, E, num_nodes=N if with_nodes else 0)
    ctx = Context(R, E, K, T, 64, num_channels=8, num_nodes=N)
    ref = ctx.get_dispatch_layout(idxd, nodes=with_nodes)
    torch.cuda.synchronize()
    for call in range(2):
        got, status = _noalloc(lib, R, E, K, T, N, idxd, with_nodes)
        assert status == 0
        for k in KEYS + (NODE_KEYS if with_nodes else ()):
            eq(got[k], exp[k], f"call {call}: {k} against the oracle")
            assert torch.equal(got[k], ref[k]), (call, k)


def test_noalloc_flags_out_of_range_expert_and_keeps_the_rest_exact():
    """An expert index outside [-1, E) is skipped and reported as bit 1 of
    status_out; every other entry is counted as usual (the oracle's layout of
    the same routing with that entry masked)."""
    lib = _lib.load()
    R, E, K, T, N = 8, 64, 4, 300, 2
    idx = inputs.random_topk(R, E, K, T, 5, 0.05)
    bad = idx.clone()
    bad[3, 17, 2] = E          # one past the last expert
    bad[6, 299, 0] = -5        # below the mask value
    masked = bad.clone()
    masked[3, 17, 2] = -1
    masked[6, 299, 0] = -1
    exp = orc.layout(masked, R, E, num_nodes=N)
    for call in range(2):
        got, status = _noalloc(lib, R, E, K, T, N, bad.cuda(), True)
        assert status == 1, status
        for k in KEYS + NODE_KEYS:
            eq(got[k], exp[k], f"call {call}: {k}")
    # a valid routing right after: the status is clean again
    got, status = _noalloc(lib, R, E, K, T, N, masked.cuda(), True)
    assert status == 0
    for k in KEYS + NODE_KEYS:
        eq(got[k], exp[k], k)


def test_noalloc_without_status_out():
    """status_out may be NULL: the outputs are the same."""
    lib = _lib.load()
    R, E, K, T, N = 16, 256, 8, 513, 4
    idx = inputs.random_topk(R, E, K, T, 7, 0.02)
    exp = orc.layout(idx, R, E, num_nodes=N)
    for call in range(2):
        got, _ = _noalloc(lib, R, E, K, T, N, idx.cuda(), True, with_status=False)
        for k in KEYS + NODE_KEYS:
            eq(got[k], exp[k], f"call {call}: {k}")


def test_noalloc_rejects_oversized_problems():
    lib = _lib.load()
    R, E, K, T = 64, 4096, 8, 10000  # needs about 40 MB of scratch
    idx = torch.zeros(1, dtype=torch.int64, device="cuda")
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = lib.ep_get_dispatch_layout_noalloc(R, E, K, T, 1, _p(idx), _p(dummy), _p(dummy), _p(dummy), None, None,
                                            None, None)
    assert rc == -3
    assert b"scratch" in lib.ep_last_error()


def test_noalloc_scratch_boundary():
    """The largest problem the fixed scratch holds runs and matches the
    oracle; one more tile is rejected with EP_ERR_CAPACITY.  R=8, E=256, no
    node outputs: the scratch needs 4 * (128 + 8 * ceil(T / 256) * 264) bytes,
    at most 1 MiB up to T = 124 * 256."""
    lib = _lib.load()
    R, E, K = 8, 256, 8
    T = 124 * 256
    assert 4 * (128 + R * (T // 256) * (E + R)) <= 1 << 20 < 4 * (128 + R * (T // 256 + 1) * (E + R))
    idx = inputs.random_topk(R, E, K, T, 9, 0.01)
    exp = orc.layout(idx, R, E)
    got, status = _noalloc(lib, R, E, K, T, 1, idx.cuda(), False)
    assert status == 0
    for k in KEYS:
        eq(got[k], exp[k], k)
    T2 = T + 1
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    idx2 = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = lib.ep_get_dispatch_layout_noalloc(R, E, K, T2, 1, _p(idx2), _p(dummy), _p(dummy), _p(dummy), None, None,
                                            None, None)
    assert rc == -3
