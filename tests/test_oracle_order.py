"""Closed-form pins of the combine's fp32 order, built so that the order shows
through the bf16 output (random data almost never does: bf16 rounding hides
fp32-level differences).

* Rank order: partials 2^25, -2^25 and 1 on ranks 0, 1, 2.  In rank order
  (2^25 - 2^25) + 1 = 1; in any order that adds 1 to -2^25 first the 1 is lost
  (fp32 spacing at 2^25 is 4) and the result is 0.
* Fused multiply-add: two experts on one rank with weights (1 + 2^-23) and
  -(1 + 2^-23) on x = 1.5.  fma keeps the rounding residual of the first
  product (non-zero); a separately rounded multiply and add cancels to 0.
* Hierarchical grouping: partials 2^25 on node 0, -2^25 and 1 on node 1: the
  node partial -2^25 + 1 loses the 1, so the three-level sum is 0 while the
  flat rank order gives 1.
"""
from fractions import Fraction

import numpy as np
import torch

import pyref

R, E, K, T, H, N = 4, 8, 4, 1, 8, 2  # L = 2 experts per rank, G = 2 ranks per node


def _run(orc, experts, weights, xval):
    idx = np.full((R, T, K), -1, np.int64)
    w = np.zeros((R, T, K), np.float32)
    idx[0, 0, :len(experts)] = experts
    w[0, 0, :len(weights)] = weights
    x = torch.full((R, T, H), xval, dtype=torch.float32).to(torch.bfloat16)
    lay = orc.layout(idx, R, E)
    note = orc.notify(lay, R, E, T, 1)
    disp = orc.dispatch(x, idx, w, note, R, E)
    perm = orc.permute(idx, disp["recv_x"], note, R, E)
    flat = orc.combine(perm["permuted_x"], perm["perm_pos"], idx, w, R, E, "ord32")[0, 0]
    hier = orc.combine_hier(perm["permuted_x"], perm["perm_pos"], idx, w, R, E, N)[0, 0]
    return flat, hier


def test_rank_partials_summed_in_rank_order(orc):
    big = float(2 ** 25)
    # experts 0, 2, 4 live on ranks 0, 1, 2
    flat, _ = _run(orc, [0, 2, 4], [big, -big, 1.0], 1.0)
    assert (flat == pyref.bf16_bits_of(1.0)).all()
    # the same partials in another rank order: 1 on rank 0, 2^25 on rank 1, -2^25 on rank 2
    flat2, _ = _run(orc, [0, 2, 4], [1.0, big, -big], 1.0)
    assert (flat2 == pyref.bf16_bits_of(0.0)).all()  # (1 + 2^25) - 2^25 = 0 in fp32


def test_rank_partial_is_a_fused_multiply_add_chain(orc):
    w0 = float(np.float32(1.0 + 2.0 ** -23))
    flat, _ = _run(orc, [0, 1], [w0, -w0], 1.5)  # experts 0 and 1 both on rank 0
    # exact expectation: fma(-w0, 1.5, round(w0 * 1.5))
    r = pyref.round_f32(Fraction(w0) * Fraction(3, 2))
    exp = pyref.fmaf(-w0, 1.5, r)
    assert exp != 0.0
    assert (flat == pyref.bf16_bits_of(exp)).all()


def test_hierarchical_grouping(orc):
    big = float(2 ** 25)
    # expert 0 on rank 0 (node 0); experts 4, 6 on ranks 2, 3 (node 1)
    flat, hier = _run(orc, [0, 4, 6], [big, -big, 1.0], 1.0)
    assert (flat == pyref.bf16_bits_of(1.0)).all()
    assert (hier == pyref.bf16_bits_of(0.0)).all()
