"""The oracle against the hand-derived worked case (R=4, E=8, EP=4, topk=2)."""
import numpy as np
import pytest

from golden_io import load

G = load("worked_r4e8.txt")
R, E, K, T, C, N, CAP = (int(G[k]) for k in ("R", "E", "K", "T", "C", "N", "ll_cap"))
L = E // R


def _topk():
    idx = np.full((R, T, K), -1, np.int64)
    idx[0] = G["topk_idx[0]"].astype(np.int64)
    return idx


def _x(H=128):
    rng = np.random.default_rng(5)
    import torch
    return torch.from_numpy(rng.standard_normal((R, T, H)).astype(np.float32)).to(torch.bfloat16)


def _w():
    import torch
    rng = np.random.default_rng(6)
    return torch.from_numpy(rng.random((R, T, K)).astype(np.float32))


@pytest.fixture(scope="module")
def chain(orc):
    idx = _topk()
    lay = orc.layout(idx, R, E, num_nodes=N)
    note = orc.notify(lay, R, E, T, C)
    x, w = _x(), _w()
    disp = orc.dispatch(x, idx, w, note, R, E)
    perm = orc.permute(idx, disp["recv_x"], note, R, E)
    return dict(idx=idx, lay=lay, note=note, disp=disp, perm=perm, x=x, w=w)


def test_layout(chain):
    lay = chain["lay"]
    np.testing.assert_array_equal(lay["num_tokens_per_expert"][0], G["num_tokens_per_expert[0]"])
    np.testing.assert_array_equal(lay["num_tokens_per_rank"][0], G["num_tokens_per_rank[0]"])
    np.testing.assert_array_equal(lay["is_token_in_rank"][0], G["is_token_in_rank[0]"])
    assert lay["num_tokens_per_expert"][1:].sum() == 0
    assert lay["is_token_in_rank"][1:].sum() == 0
    np.testing.assert_array_equal(lay["num_tokens_per_node"][0], G["num_tokens_per_node[0]"])
    np.testing.assert_array_equal(lay["is_token_in_node"][0], G["is_token_in_node[0]"])


def test_notify(chain):
    n = chain["note"]
    for key in ("recv_count", "num_recv_tokens", "recv_offsets", "rank_base", "num_recv_per_expert",
                "expert_offsets", "perm_rank_base"):
        np.testing.assert_array_equal(n[key], G[key], err_msg=key)
    np.testing.assert_array_equal(n["channel_prefix_matrix"][0], G["channel_prefix_matrix[0]"])
    assert (n["channel_prefix_matrix"][1:] == 0).all()
    np.testing.assert_array_equal(n["send_pos"][0], G["send_pos[0]"])
    assert (n["send_pos"][1:] == -1).all()


def test_dispatch_and_permute(chain):
    d, p, x = chain["disp"], chain["perm"], chain["x"]
    xb = x.view(__import__("torch").int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(d["recv_src_rank"], np.zeros(6))
    np.testing.assert_array_equal(d["recv_src_idx"], G["recv_src_idx"])
    np.testing.assert_array_equal(d["recv_topk_idx"], G["recv_topk_idx"])
    for r, t in enumerate(G["recv_src_idx"].astype(int)):
        np.testing.assert_array_equal(d["recv_x"][r], xb[0, t])
    np.testing.assert_array_equal(p["perm_src_row"], G["perm_src_row"])
    np.testing.assert_array_equal(p["perm_pos"][0], G["perm_pos[0]"])
    # rank 3 receives (t2, t3) but its permuted block is (expert 6: t3, expert 7: t2)
    np.testing.assert_array_equal(d["recv_x"][4], xb[0, 2])
    np.testing.assert_array_equal(p["permuted_x"][5], xb[0, 3])
    np.testing.assert_array_equal(p["permuted_x"][6], xb[0, 2])
    # rank 0 holds two copies of token 0, for experts 0 and 1
    np.testing.assert_array_equal(p["permuted_x"][0], xb[0, 0])
    np.testing.assert_array_equal(p["permuted_x"][1], xb[0, 0])


def test_low_latency(orc, chain):
    x, idx = chain["x"], chain["idx"]
    sent = orc.ll_send(x, idx, R, E, CAP)
    counts = sent["counts"]
    np.testing.assert_array_equal(counts[:, 0], G["ll_counts_src0"])
    assert (counts[:, 1:] == 0).all()
    np.testing.assert_array_equal(sent["slot"][0], G["ll_slot[0]"])
    m = int(G["ll_region_e7_s0"])
    assert m == (7 * R + 0) * CAP
    assert sent["reg_src"][m] == 2  # token 2 is expert 7's only sender
    pk = orc.ll_pack(sent, R, E, 128, CAP)
    np.testing.assert_array_equal(pk["packed_recv_count"], G["packed_recv_count"])


def test_hier_stage_pos(orc, chain):
    sb, sp = orc.hier_stage_pos(chain["lay"], R, T, N)
    np.testing.assert_array_equal(sb, G["stage_base"])
    np.testing.assert_array_equal(sp[0], G["stage_pos[0]"])
    assert (sp[1:] == -1).all()
