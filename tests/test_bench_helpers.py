"""Host-side arithmetic of bench.py: algorithmic bytes per kernel, the
percentile helper and the nominal-bandwidth percentages (no GPU)."""
import bench


def test_algo_bytes_prefill_shape():
    H, K = 7168, 8
    tokens, copies, pairs = 32768, 175243, 262144
    ab = bench.algo_bytes(H, K, tokens, copies, pairs)
    row = 2 * H
    assert ab["dispatch"] == (tokens + copies) * row            # x read once, one row per copy written
    assert ab["permute"] == (copies + pairs) * row              # each received row read once, one row per pair
    assert ab["combine"] == (pairs + tokens) * row + tokens * K * 8
    # staged (hierarchical): stage rows are written once and read once more
    st = bench.algo_bytes(H, K, tokens, copies, pairs, staged=1000)
    assert st["dispatch"] - ab["dispatch"] == 2 * 1000 * row


def test_ll_algo_bytes():
    H, tokens, pairs = 7168, 2048, 16384
    lb = bench.ll_algo_bytes(H, tokens, pairs)
    msg = H + H // 32 + 4
    assert lb["ll_send"] == tokens * 2 * H + pairs * msg
    assert lb["ll_recv"] == 2 * pairs * msg


def test_percentile_and_nominal_pct():
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.pct(xs, 0.0) == 1.0 and bench.pct(xs, 0.5) == 3.0 and bench.pct(xs, 1.0) == 5.0
    d = bench.add_nominal_pct({"effective_GBps": 6000.0,
                               "kernels": {"a": {"GBps": 4000.0, "frac": 0.59}},
                               "legs": [{"GBps": 800.0}]})
    assert d["effective_pct_of_8TBps"] == 75.0
    assert d["kernels"]["a"]["pct_of_8TBps"] == 50.0 and d["kernels"]["a"]["frac"] == 0.59
    assert d["legs"][0]["pct_of_8TBps"] == 10.0
