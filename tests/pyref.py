"""An independent, dictionary-based Python formulation of the dispatch / combine
definitions, used only to brute-force the C oracle on tiny inputs.

It is deliberately written another way from the oracle (sorted lists and
dicts keyed by tuples instead of running counters), so that a mistake in one
is unlikely to be repeated in the other.
"""
from fractions import Fraction
import math
import struct

import numpy as np


def layout(idx, R, E, N=0):
    Rr, T, K = idx.shape
    L = E // R
    G = R // N if N else 1
    valid = {(s, t, k): int(idx[s, t, k]) for s in range(R) for t in range(T) for k in range(K)
             if idx[s, t, k] >= 0}
    ntpe = np.zeros((R, E), np.int64)
    for (s, t, k), e in valid.items():
        ntpe[s, e] += 1
    ranks_of = {}
    for (s, t, k), e in valid.items():
        ranks_of.setdefault((s, t), set()).add(e // L)
    itir = np.zeros((R, T, R), np.int64)
    for (s, t), ds in ranks_of.items():
        for d in ds:
            itir[s, t, d] = 1
    ntpr = itir.sum(axis=1)
    out = dict(num_tokens_per_expert=ntpe, num_tokens_per_rank=ntpr, is_token_in_rank=itir)
    if N:
        itin = np.zeros((R, T, N), np.int64)
        for (s, t), ds in ranks_of.items():
            for d in ds:
                itin[s, t, d // G] = 1
        out["is_token_in_node"] = itin
        out["num_tokens_per_node"] = itin.sum(axis=1)
    return out, valid


def receive_lists(itir):
    """For each receiver d, the list of (s, t) it receives, in (s, t) order."""
    R, T, _ = itir.shape
    return {d: sorted((s, t) for s in range(R) for t in range(T) if itir[s, t, d]) for d in range(R)}


def send_pos(itir):
    R, T, _ = itir.shape
    lists = receive_lists(itir)
    sp = -np.ones((R, T, R), np.int64)
    for d, lst in lists.items():
        for i, (s, t) in enumerate(lst):
            sp[s, t, d] = i
    return sp, lists


def channel_prefix(itir, C):
    R, T, _ = itir.shape
    ct = -(-T // C) if T else 0
    cpm = np.zeros((R, R, C), np.int64)
    for s in range(R):
        for d in range(R):
            for c in range(C):
                hi = min(T, (c + 1) * ct)
                cpm[s, d, c] = sum(int(itir[s, t, d]) for t in range(0, hi))
    return cpm


def permute_order(valid, R, E):
    """Pairs sorted by (rank, local expert, s, t, k) -> global permuted index."""
    L = E // R
    keys = sorted(((e // L, e % L, s, t, k) for (s, t, k), e in valid.items()))
    return {(s, t, k): i for i, (d, l, s, t, k) in enumerate(keys)}, keys


def ll_slots(valid, R, E, T, K, t0, n):
    """slot of (s, t, k): its index among entries of source s for expert e in (t, k) order."""
    groups = {}
    for (s, t, k), e in sorted(valid.items()):
        if t0 <= t < t0 + n:
            groups.setdefault((s, e), []).append((t, k))
    slot = {}
    for (s, e), lst in groups.items():
        for i, (t, k) in enumerate(lst):
            slot[(s, t, k)] = i
    counts = {(s, e): len(lst) for (s, e), lst in groups.items()}
    return slot, counts


def stage_positions(itin, R, N):
    Rr, T, _ = itin.shape
    G = R // N
    rows = []
    for h in range(R):
        n = h // G
        srcs = [s for s in range(R) if s % G == h % G]
        for s in srcs:
            for t in range(T):
                if itin[s, t, n]:
                    rows.append((h, s, t, n))
    pos = {(s, t, n): i for i, (h, s, t, n) in enumerate(rows)}
    base = [0] * (R + 1)
    for h in range(R):
        base[h + 1] = base[h] + sum(1 for r in rows if r[0] == h)
    return pos, base


# ---------------------------------------------------------------------------
# exact fp32 arithmetic for tiny combine checks
# ---------------------------------------------------------------------------

def _f32(v: float) -> float:
    return struct.unpack("<f", struct.pack("<f", v))[0]


def _f32_neighbours(x: float):
    b = struct.unpack("<I", struct.pack("<f", x))[0]
    out = [x]
    for nb in (b - 1, b + 1):
        if 0 <= nb < 2 ** 32:
            v = struct.unpack("<f", struct.pack("<I", nb))[0]
            if math.isfinite(v):
                out.append(v)
    return out


def round_f32(q: Fraction) -> float:
    """Exact value -> nearest fp32, ties to the even significand."""
    if q == 0:
        return 0.0
    approx = _f32(float(q))
    cands = set()
    for c in _f32_neighbours(approx):
        cands.update(_f32_neighbours(c))
    best = None
    for c in cands:
        dist = abs(Fraction(c) - q)
        if best is None or dist < best[0]:
            best = (dist, [c])
        elif dist == best[0]:
            best[1].append(c)
    choices = best[1]
    if len(choices) == 1:
        return choices[0]
    even = [c for c in choices if struct.unpack("<I", struct.pack("<f", c))[0] % 2 == 0]
    return even[0]


def fmaf(a: float, b: float, c: float) -> float:
    """fp32 fused multiply-add: one rounding of the exact a*b + c."""
    exact = Fraction(a) * Fraction(b) + Fraction(c)
    if exact != 0:
        return round_f32(exact)
    prod_neg = math.copysign(1.0, a) * math.copysign(1.0, b) < 0
    if (a == 0 or b == 0) and c == 0:
        return -0.0 if (prod_neg and math.copysign(1.0, c) < 0) else 0.0
    return 0.0


def fadd(a: float, b: float) -> float:
    exact = Fraction(a) + Fraction(b)
    if exact != 0:
        return round_f32(exact)
    if a == 0 and b == 0 and math.copysign(1.0, a) < 0 and math.copysign(1.0, b) < 0:
        return -0.0
    return 0.0


def bf16_bits_of(v) -> int:
    """Exact value -> bits of the nearest bf16, ties to the even significand,
    by comparing distances to the bracketing bf16 values."""
    q = Fraction(v)
    if q == 0:
        return 0x8000 if (isinstance(v, float) and math.copysign(1.0, v) < 0) else 0
    neg = q < 0
    a = -q if neg else q
    # bracket a between consecutive positive bf16 values lo <= a < hi
    lo_bits, hi_bits = 0, 0x7F80
    while hi_bits - lo_bits > 1:
        mid = (lo_bits + hi_bits) // 2
        if Fraction(bf16_value(mid)) <= a:
            lo_bits = mid
        else:
            hi_bits = mid
    dlo = a - Fraction(bf16_value(lo_bits))
    dhi = Fraction(bf16_value(hi_bits)) - a if hi_bits < 0x7F80 else None
    if dhi is None or dlo < dhi or (dlo == dhi and lo_bits % 2 == 0):
        bits = lo_bits
    else:
        bits = hi_bits
    return bits | (0x8000 if neg else 0)


def bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


# ---------------------------------------------------------------------------
# low-latency pack and combine, written from the definitions
# ---------------------------------------------------------------------------

def ll_packed_rows(valid, R, E, T, K, t0, n):
    """Where every valid (s, t, k) of the microbatch [t0, t0 + n) sits in the
    packed per-expert layout: {(s, t, k): (d, l, row)}, row counted inside
    expert (d, l)'s block.  Sources are laid out one after another in s order,
    and inside a source the entries keep their (t, k) order."""
    L = E // R
    slot, counts = ll_slots(valid, R, E, T, K, t0, n)
    where = {}
    for (s, t, k), i in slot.items():
        e = valid[(s, t, k)]
        before = sum(counts.get((s2, e), 0) for s2 in range(s))
        where[(s, t, k)] = (e // L, e % L, before + i)
    return where


def ll_combine_exact(y_rows, where, idx, w, t0, n):
    """out[s][t] as exact bf16 bits: for k ascending over the valid entries,
    acc = fma(w, y, acc) rounded once to fp32 per step, then bf16 (nearest,
    ties to even).  y_rows maps (d, l, row) to a list of fp32 values (one per
    channel); returns {(s, t): [bits per channel]} for tokens of the batch."""
    R, T, K = idx.shape
    out = {}
    H = len(next(iter(y_rows.values()))) if y_rows else 0
    for s in range(R):
        for t in range(t0, t0 + n):
            ks = [k for k in range(K) if (s, t, k) in where]
            vals = []
            for j in range(H):
                acc = 0.0
                for k in ks:
                    acc = fmaf(float(w[s, t, k]), y_rows[where[(s, t, k)]][j], acc)
                vals.append(bf16_bits_of(acc))
            out[(s, t)] = vals
    return out
