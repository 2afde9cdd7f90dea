"""The oracle's number formats against torch's casts and closed forms.

e4m3 (OCP FP8, the format of the low-latency dispatch on the page
"事件驱动 EP 内核的调度策略与零拷贝通信", section "低延迟模式": FP8 dispatch, BF16
combine) and bf16 rounding."""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import pyref


def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_every_bf16_value_in_range(orc):
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 464.0)]
    np.testing.assert_array_equal(orc.e4m3_encode(v), _torch_e4m3(v))


def test_e4m3_random_quotients(orc):
    """Quotients x / (amax / 448) of random bf16 blocks, as the quantiser makes them."""
    rng = np.random.default_rng(0)
    xs = torch.from_numpy(rng.standard_normal((400, 128)).astype(np.float32) *
                          np.exp(rng.uniform(-8, 8, (400, 1))).astype(np.float32)).to(torch.bfloat16).float()
    amax = xs.abs().amax(dim=1, keepdim=True)
    scale = amax / 448.0
    q = (xs / scale).numpy()
    np.testing.assert_array_equal(orc.e4m3_encode(q), _torch_e4m3(q))


def test_e4m3_ties_and_subnormals(orc):
    vals = []
    for c in range(0, 0x7E):  # consecutive positive finite codes
        a, b = orc.e4m3_decode(c), orc.e4m3_decode(c + 1)
        vals += [a, b, (a + b) / 2, np.nextafter(np.float32((a + b) / 2), np.float32(0)),
                 np.nextafter(np.float32((a + b) / 2), np.float32(1000))]
    v = np.array(vals, np.float32)
    v = np.concatenate([v, -v])
    np.testing.assert_array_equal(orc.e4m3_encode(v), _torch_e4m3(v))
    # ties go to the even code: midway between codes 1 and 2 (subnormal) is 1.5 * 2^-9
    assert orc.e4m3_encode(np.array([1.5 * 2.0 ** -9], np.float32))[0] == 2
    assert orc.e4m3_encode(np.array([0.5 * 2.0 ** -9], np.float32))[0] == 0
    # smallest normal 2^-6 is code 0x08; largest subnormal is 7 * 2^-9
    assert orc.e4m3_encode(np.array([2.0 ** -6], np.float32))[0] == 0x08
    assert orc.e4m3_encode(np.array([7 * 2.0 ** -9], np.float32))[0] == 0x07


def test_e4m3_saturation_and_signs(orc):
    v = np.array([448.0, 449.0, 464.0, 480.0, 1e9, np.inf, -448.0, -1e9, -np.inf, -0.0, 0.0], np.float32)
    np.testing.assert_array_equal(orc.e4m3_encode(v),
                                  [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0xFE, 0x80, 0x00])
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert math.isnan(orc.e4m3_decode(0x7F))


def test_decode_matches_torch(orc):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([orc.e4m3_decode(int(c)) for c in codes], np.float32)
    np.testing.assert_array_equal(got, ref)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_quantize_row_closed_forms(orc):
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal((1, 1024)).astype(np.float32) * 2)
    xb = x.view(torch.int16).numpy().view(np.uint16)[0]
    codes, scales = orc.quantize_row(xb)
    xf = x.float().numpy()[0]
    for b in range(8):
        blk = xf[b * 128:(b + 1) * 128]
        amax = np.float32(np.abs(blk).max())
        assert scales[b] == np.float32(amax / np.float32(448.0))
        j = int(np.abs(blk).argmax())
        # the element holding the block maximum encodes to +-448
        assert codes[b * 128 + j] == (0xFE if blk[j] < 0 else 0x7E)
        # dequantisation error: half an e4m3 ulp (2^-4 relative) for normals,
        # half the subnormal step (2^-10) times the scale otherwise
        deq = np.array([orc.e4m3_decode(int(c)) for c in codes[b * 128:(b + 1) * 128]], np.float64) * scales[b]
        bound = 2.0 ** -4 * np.abs(blk) + 2.0 ** -10 * scales[b]
        assert (np.abs(deq - blk) <= bound * (1 + 1e-6) + 1e-30).all()


def test_quantize_zero_block(orc):
    xb = np.zeros(256, np.uint16)
    xb[5] = 0x8000  # -0.0
    xb[130:140] = _bf16(np.linspace(-1, 1, 10)).view(torch.int16).numpy().view(np.uint16)
    codes, scales = orc.quantize_row(xb)
    assert scales[0] == 0.0
    assert codes[5] == 0x80 and codes[:5].max() == 0 and codes[6:128].max() == 0
    assert scales[1] == np.float32(np.float32(1.0) / np.float32(448.0))


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(2)
    v = rng.standard_normal(20000).astype(np.float32) * np.exp(rng.uniform(-30, 30, 20000)).astype(np.float32)
    # exact ties: bf16 value plus half its ulp
    base = _bf16(rng.standard_normal(2000).astype(np.float32)).float().numpy().astype(np.float64)
    _, ex = np.frexp(base)
    half_ulp = np.ldexp(1.0, ex - 9)  # |b| in [2^(ex-1), 2^ex): bf16 ulp is 2^(ex-8)
    ties = np.concatenate([base + half_ulp, base - half_ulp]).astype(np.float32)
    allv = np.concatenate([v, ties, np.array([0.0, -0.0, 1e-40, -3e38], np.float32)])
    ref = torch.from_numpy(allv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16(float(a)) for a in allv], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_f64_to_bf16_exact_nearest(orc):
    rng = np.random.default_rng(4)
    vals = list(rng.standard_normal(3000) * np.exp(rng.uniform(-20, 20, 3000)))
    # doubles just beside a bf16 midpoint: a cast through fp32 would round twice
    for b in rng.standard_normal(300):
        bb = pyref.bf16_value(pyref.bf16_bits_of(float(b)))
        _, ex = math.frexp(bb)
        mid = bb + math.copysign(math.ldexp(1.0, ex - 9), bb)
        vals += [mid, math.nextafter(mid, 0.0), math.nextafter(mid, math.inf)]
    for v in vals:
        assert orc.f64_to_bf16(v) == pyref.bf16_bits_of(Fraction(v)), v
