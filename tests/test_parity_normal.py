"""GPU vs oracle, element by element, for the normal path: layout, notify,
dispatch scatter, permute and combine (bit-exact; combine also within the
stated tolerance of the fp64 reference).  Sizes span several 256-token tiles,
ragged channels and tails, and the edge cases of the method."""
import pytest
import torch

from combine_get_dispatch_histograms_gb300 import inputs
from parity_util import compare_normal

pytestmark = pytest.mark.gpu

CASES = [
    # name, R, E, K, T, H, C, mask_p, distinct, seed
    ("tiny-config", None),
    ("ragged", (4, 8, 2, 600, 136, 3, 0.1, True, 1)),        # tiles + ragged channels, H not a multiple of 64
    ("eight-ranks", (8, 256, 8, 700, 512, 8, 0.0, True, 2)),
    ("masked-dups", (4, 16, 4, 333, 64, 5, 0.3, False, 3)),   # duplicates inside a token
    ("no-tokens", (4, 8, 2, 0, 64, 2, 0.0, True, 4)),
    ("all-masked", (4, 8, 2, 100, 64, 2, 1.0, True, 5)),
    ("single-rank", (1, 8, 4, 300, 64, 4, 0.1, True, 6)),
    ("one-expert-per-rank", (8, 8, 3, 257, 64, 1, 0.0, True, 7)),
    ("top1", (4, 32, 1, 513, 64, 16, 0.0, True, 8)),
    ("max-ranks-topk", (64, 128, 32, 40, 64, 8, 0.05, True, 9)),
    ("many-experts", (16, 4096, 8, 96, 64, 4, 0.0, True, 10)),
    ("more-channels-than-tokens", (4, 8, 2, 5, 64, 64, 0.0, True, 11)),
    ("rows-in-chunks", (4, 16, 4, 50, 16384, 4, 0.1, True, 14)),       # 32 KB rows: several bulk chunks per row
    ("ragged-chunk", (4, 8, 2, 40, 12296, 2, 0.0, True, 15)),          # last chunk of a row shorter
]


@pytest.mark.parametrize("name,case", CASES, ids=[c[0] for c in CASES])
def test_normal_path(name, case):
    if case is None:
        w = inputs.WORKLOADS["tiny"]
        x, idx, wts = inputs.make_inputs(w, seed=0)
        compare_normal(w.R, w.E, w.K, w.T, w.H, w.num_channels, x, idx, wts)
        return
    R, E, K, T, H, C, mask_p, distinct, seed = case
    idx = inputs.random_topk(R, E, K, T, seed, mask_p, distinct)
    x = inputs.random_x(R, T, H, seed)
    wts = inputs.random_weights(R, T, K, seed)
    compare_normal(R, E, K, T, H, C, x, idx, wts)


def test_hot_expert_and_single_receiver():
    """Every token routes to experts of rank 0 only (skew at its worst)."""
    R, E, K, T, H = 8, 64, 4, 400, 64
    g = torch.Generator().manual_seed(12)
    idx = torch.stack([torch.randperm(8, generator=g)[:K] for _ in range(R * T)]).reshape(R, T, K).to(torch.int64)
    x = inputs.random_x(R, T, H, 12)
    wts = inputs.random_weights(R, T, K, 12)
    compare_normal(R, E, K, T, H, 4, x, idx, wts)


def test_repeatable_calls_same_context():
    """Completion counters re-arm: two calls on one context give the same result."""
    from parity_util import run_gpu_normal, bits
    R, E, K, T, H = 4, 16, 4, 300, 64
    idx = inputs.random_topk(R, E, K, T, 13, 0.1)
    x = inputs.random_x(R, T, H, 13)
    wts = inputs.random_weights(R, T, K, 13)
    a = run_gpu_normal(R, E, K, T, H, 4, x, idx, wts)
    b = run_gpu_normal(R, E, K, T, H, 4, x, idx, wts)
    assert (bits(a[5]) == bits(b[5])).all()
    ctx = a[0]
    lay1 = ctx.get_dispatch_layout(idx.cuda())
    lay2 = ctx.get_dispatch_layout(idx.cuda())
    for k in lay1:
        assert torch.equal(lay1[k], lay2[k])
