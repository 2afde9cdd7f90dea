"""Plain CPU oracle for MoE expert-parallel dispatch / combine.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's
CPU-baseline leg are the only code that may import this package.  It shares
no code with the CUDA path (its arithmetic lives in ``ep_oracle.c``, a scalar
C restatement of each step's definition; this module only marshals numpy
arrays through ctypes).

Pinned by the not-gpu tests in ``tests/test_oracle_*.py``: a hand-derived worked
case, invariants, brute force against an independent Python formulation, the
e4m3 codec against ``torch.float8_e4m3fn`` and closed forms.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_HDR = os.path.join(_HERE, "ep_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libep_oracle.so")
_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_SO) and \
            os.path.getmtime(_SO) >= max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    """The oracle library.  EP_ORACLE_LIB names another build of ep_oracle.c
    (the mutation tests load deliberately broken copies through it)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("EP_ORACLE_LIB") or build()
            _lib = ctypes.CDLL(path)
            _declare(_lib)
    return _lib


def _declare(L):
    sig = {
        "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
        "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "orc_e4m3_decode": (ctypes.c_float, [ctypes.c_uint8]),
        "orc_e4m3_encode_array": (None, [P, P, I64]),
        "orc_quantize_row": (None, [P, I, P, P]),
        "orc_layout": (I, [I, I, I, I, I, P, P, P, P, P, P]),
        "orc_notify": (I, [I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P]),
        "orc_dispatch": (I, [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P]),
        "orc_permute": (I, [I, I, I, I, I, P, P, P, P, P, P, P]),
        "orc_notify_aligned": (I, [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P]),
        "orc_permute_aligned": (I, [I, I, I, I, I, I, ctypes.c_int64, P, P, P, P, P, P, P]),
        "orc_combine_ord32": (I, [I, I, I, I, I, P, P, P, P, P]),
        "orc_combine_ref64": (I, [I, I, I, I, I, P, P, P, P, P]),
        "orc_ll_send": (I, [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P]),
        "orc_ll_pack": (I, [I, I, I, I, P, P, P, P, P, P, P, P, P]),
        "orc_ll_combine": (I, [I, I, I, I, I, I, I, I, P, P, P, P, P, P]),
        "orc_ll_dequant": (I, [I, I, P, P, P]),
        "orc_hier_stage_pos": (I, [I, I, I, P, P, P, P]),
        "orc_hier_stage_a": (I, [I, I, I, I, P, P, P, P, P]),
        "orc_hier_stage_b": (I, [I, I, I, I, I, P, P, P, P, P, P, P, P]),
        "orc_combine_hier_ord32": (I, [I, I, I, I, I, I, P, P, P, P, P]),
        "orc_ll_message_bytes": (I64, [I]),
        "orc_ll_size_hint": (I64, [I, I, I, I]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


# ---------------------------------------------------------------------------
# array helpers
# ---------------------------------------------------------------------------

def _np(a, dtype):
    """Contiguous numpy view of a torch CPU tensor or numpy array."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.int16)
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        if dtype == np.uint16 and a.dtype == np.int16:
            a = a.view(np.uint16)
        elif dtype == np.uint8 and a.dtype in (np.bool_, np.int8):
            a = a.view(np.uint8) if a.dtype == np.int8 else a.astype(np.uint8)
        else:
            a = a.astype(dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def bf16_bits(x) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (numpy)."""
    return _np(x, np.uint16)


class OracleError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {code}")
        self.code = code


def _ok(fn, rc):
    if rc != 0:
        raise OracleError(fn, rc)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def e4m3_encode(v) -> np.ndarray:
    v = _np(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(v), _p(out), v.size)
    return out


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def f32_to_bf16(v: float) -> int:
    return lib().orc_f32_to_bf16(float(v))


def f64_to_bf16(v: float) -> int:
    return lib().orc_f64_to_bf16(float(v))


def quantize_row(x_bits: np.ndarray):
    x_bits = _np(x_bits, np.uint16)
    H = x_bits.shape[-1]
    codes = np.empty(H, np.uint8)
    scales = np.empty(H // 128, np.float32)
    lib().orc_quantize_row(_p(x_bits), H, _p(codes), _p(scales))
    return codes, scales


def quantize_rows(x_bits: np.ndarray):
    """quantize_row over every row of a [N][H] array (a loop of single-row
    calls: the codes and scales of each row depend on that row alone)."""
    x_bits = _np(x_bits, np.uint16)
    n, H = x_bits.shape
    codes = np.empty((n, H), np.uint8)
    scales = np.empty((n, H // 128), np.float32)
    f = lib().orc_quantize_row
    for i in range(n):
        f(_p(x_bits[i]), H, _p(codes[i]), _p(scales[i]))
    return codes, scales


# ---------------------------------------------------------------------------
# normal (high-throughput) mode
# ---------------------------------------------------------------------------

def layout(topk_idx, R: int, E: int, num_nodes: int = 0):
    idx = _np(topk_idx, np.int64)
    Rr, T, K = idx.shape
    assert Rr == R
    out = dict(
        num_tokens_per_expert=np.empty((R, E), np.int32),
        num_tokens_per_rank=np.empty((R, R), np.int32),
        is_token_in_rank=np.empty((R, T, R), np.uint8),
    )
    ntpn = itin = None
    if num_nodes > 0:
        ntpn = np.empty((R, num_nodes), np.int32)
        itin = np.empty((R, T, num_nodes), np.uint8)
        out["num_tokens_per_node"] = ntpn
        out["is_token_in_node"] = itin
    rc = lib().orc_layout(R, E, K, T, num_nodes, _p(idx), _p(out["num_tokens_per_expert"]),
                          _p(out["num_tokens_per_rank"]), _p(out["is_token_in_rank"]), _p(ntpn), _p(itin))
    _ok("orc_layout", rc)
    return out


def notify(lay: dict, R: int, E: int, T: int, C: int, align: int = 1):
    L = E // R
    o = dict(
        recv_count=np.empty((R, R), np.int32),
        num_recv_tokens=np.empty(R, np.int32),
        recv_offsets=np.empty((R, R), np.int32),
        rank_base=np.empty(R + 1, np.int32),
        num_recv_per_expert=np.empty((R, L), np.int32),
        expert_offsets=np.empty((R, L), np.int32),
        perm_rank_base=np.empty(R + 1, np.int32),
        channel_prefix_matrix=np.empty((R, R, C), np.int32),
        send_pos=np.empty((R, T, R), np.int32),
    )
    ntpe = _np(lay["num_tokens_per_expert"], np.int32)
    ntpr = _np(lay["num_tokens_per_rank"], np.int32)
    itir = _np(lay["is_token_in_rank"], np.uint8)
    if align == 1:
        rc = lib().orc_notify(R, E, T, C, _p(ntpe), _p(ntpr), _p(itir), _p(o["recv_count"]),
                              _p(o["num_recv_tokens"]), _p(o["recv_offsets"]), _p(o["rank_base"]),
                              _p(o["num_recv_per_expert"]), _p(o["expert_offsets"]),
                              _p(o["perm_rank_base"]), _p(o["channel_prefix_matrix"]), _p(o["send_pos"]))
    else:
        rc = lib().orc_notify_aligned(R, E, T, C, align, _p(ntpe), _p(ntpr), _p(itir), _p(o["recv_count"]),
                                      _p(o["num_recv_tokens"]), _p(o["recv_offsets"]), _p(o["rank_base"]),
                                      _p(o["num_recv_per_expert"]), _p(o["expert_offsets"]),
                                      _p(o["perm_rank_base"]), _p(o["channel_prefix_matrix"]), _p(o["send_pos"]))
    _ok("orc_notify", rc)
    o["align"] = align
    return o


def dispatch(x, topk_idx, topk_weights, note: dict, R: int, E: int):
    xb = _np(x, np.uint16)
    idx = _np(topk_idx, np.int64)
    w = _np(topk_weights, np.float32)
    _, T, H = xb.shape
    K = idx.shape[2]
    n = int(note["rank_base"][R])
    o = dict(
        recv_x=np.zeros((n, H), np.uint16),
        recv_src_rank=np.empty(n, np.int32),
        recv_src_idx=np.empty(n, np.int32),
        recv_topk_idx=np.empty((n, K), np.int32),
        recv_topk_weights=np.empty((n, K), np.float32),
    )
    rc = lib().orc_dispatch(R, E, K, T, H, _p(xb), _p(idx), _p(w), _p(_np(note["send_pos"], np.int32)),
                            _p(_np(note["rank_base"], np.int32)), _p(o["recv_x"]), _p(o["recv_src_rank"]),
                            _p(o["recv_src_idx"]), _p(o["recv_topk_idx"]), _p(o["recv_topk_weights"]))
    _ok("orc_dispatch", rc)
    return o


def permute(topk_idx, recv_x, note: dict, R: int, E: int):
    idx = _np(topk_idx, np.int64)
    rx = _np(recv_x, np.uint16)
    _, T, K = idx.shape
    H = rx.shape[1]
    P = int(note["perm_rank_base"][R])
    o = dict(
        permuted_x=np.zeros((P, H), np.uint16),
        perm_src_row=np.empty(P, np.int32),
        perm_pos=np.empty((R, T, K), np.int32),
    )
    align = int(note.get("align", 1))
    if align == 1:
        rc = lib().orc_permute(R, E, K, T, H, _p(idx), _p(rx), _p(_np(note["rank_base"], np.int32)),
                               _p(_np(note["send_pos"], np.int32)), _p(o["permuted_x"]), _p(o["perm_src_row"]),
                               _p(o["perm_pos"]))
    else:
        rc = lib().orc_permute_aligned(R, E, K, T, H, align, P, _p(idx), _p(rx),
                                       _p(_np(note["rank_base"], np.int32)), _p(_np(note["send_pos"], np.int32)),
                                       _p(o["permuted_x"]), _p(o["perm_src_row"]), _p(o["perm_pos"]))
    _ok("orc_permute", rc)
    return o


def combine(expert_out, perm_pos, topk_idx, topk_weights, R: int, E: int, mode: str = "ord32"):
    y = _np(expert_out, np.uint16)
    pp = _np(perm_pos, np.int32)
    idx = _np(topk_idx, np.int64)
    w = _np(topk_weights, np.float32)
    _, T, K = idx.shape
    H = y.shape[1]
    out = np.empty((R, T, H), np.uint16)
    fn = {"ord32": lib().orc_combine_ord32, "ref64": lib().orc_combine_ref64}[mode]
    rc = fn(R, E, K, T, H, _p(y), _p(pp), _p(idx), _p(w), _p(out))
    _ok("orc_combine_" + mode, rc)
    return out


def combine_hier(expert_out, perm_pos, topk_idx, topk_weights, R: int, E: int, num_nodes: int):
    y = _np(expert_out, np.uint16)
    pp = _np(perm_pos, np.int32)
    idx = _np(topk_idx, np.int64)
    w = _np(topk_weights, np.float32)
    _, T, K = idx.shape
    H = y.shape[1]
    out = np.empty((R, T, H), np.uint16)
    rc = lib().orc_combine_hier_ord32(R, E, K, T, H, num_nodes, _p(y), _p(pp), _p(idx), _p(w), _p(out))
    _ok("orc_combine_hier_ord32", rc)
    return out


# ---------------------------------------------------------------------------
# low-latency mode
# ---------------------------------------------------------------------------

def ll_message_bytes(H: int) -> int:
    return int(lib().orc_ll_message_bytes(H))


def ll_size_hint(cap: int, H: int, R: int, E: int) -> int:
    return int(lib().orc_ll_size_hint(cap, H, R, E))


def ll_send(x, topk_idx, R: int, E: int, cap: int, t0: int = 0, n: int | None = None,
            slot: np.ndarray | None = None):
    xb = _np(x, np.uint16)
    idx = _np(topk_idx, np.int64)
    _, T, H = xb.shape
    K = idx.shape[2]
    if n is None:
        n = T - t0
    M = E * R * cap
    o = dict(
        reg_codes=np.zeros((M, H), np.uint8),
        reg_scales=np.zeros((M, H // 128), np.float32),
        reg_src=np.full(M, -1, np.int32),
        counts=np.full((E, R), -1, np.int32),
        slot=slot if slot is not None else np.full((R, T, K), -1, np.int32),
    )
    rc = lib().orc_ll_send(R, E, K, T, H, cap, t0, n, _p(xb), _p(idx), _p(o["reg_codes"]),
                           _p(o["reg_scales"]), _p(o["reg_src"]), _p(o["counts"]), _p(o["slot"]))
    _ok("orc_ll_send", rc)
    return o


def ll_pack(sent: dict, R: int, E: int, H: int, cap: int):
    L = E // R
    o = dict(
        packed_x=np.zeros((R, L, R * cap, H), np.uint8),
        packed_scales=np.zeros((R, L, R * cap, H // 128), np.float32),
        packed_src_info=np.full((R, L, R * cap, 2), -1, np.int32),
        packed_recv_count=np.empty((R, L), np.int32),
        layout_range=np.empty((R, L, R, 2), np.int32),
    )
    rc = lib().orc_ll_pack(R, E, H, cap, _p(sent["reg_codes"]), _p(sent["reg_scales"]), _p(sent["reg_src"]),
                           _p(sent["counts"]), _p(o["packed_x"]), _p(o["packed_scales"]),
                           _p(o["packed_src_info"]), _p(o["packed_recv_count"]), _p(o["layout_range"]))
    _ok("orc_ll_pack", rc)
    return o


def ll_dequant(codes, scales):
    c = _np(codes, np.uint8)
    s = _np(scales, np.float32)
    H = c.shape[-1]
    rows = c.size // H
    y = np.empty(c.shape, np.uint16)
    rc = lib().orc_ll_dequant(rows, H, _p(c), _p(s), _p(y))
    _ok("orc_ll_dequant", rc)
    return y


def ll_combine(y_ll, topk_idx, topk_weights, slot, layout_range, R: int, E: int, cap: int,
               t0: int = 0, n: int | None = None, out: np.ndarray | None = None):
    y = _np(y_ll, np.uint16)
    idx = _np(topk_idx, np.int64)
    w = _np(topk_weights, np.float32)
    sl = _np(slot, np.int32)
    lr = _np(layout_range, np.int32)
    _, T, K = idx.shape
    H = y.shape[-1]
    if n is None:
        n = T - t0
    if out is None:
        out = np.zeros((R, T, H), np.uint16)
    rc = lib().orc_ll_combine(R, E, K, T, H, cap, t0, n, _p(y), _p(idx), _p(w), _p(sl), _p(lr), _p(out))
    _ok("orc_ll_combine", rc)
    return out


# ---------------------------------------------------------------------------
# hierarchical staging
# ---------------------------------------------------------------------------

def hier_stage_pos(lay: dict, R: int, T: int, num_nodes: int):
    ntpn = _np(lay["num_tokens_per_node"], np.int32)
    itin = _np(lay["is_token_in_node"], np.uint8)
    stage_base = np.empty(R + 1, np.int32)
    stage_pos = np.empty((R, T, num_nodes), np.int32)
    rc = lib().orc_hier_stage_pos(R, T, num_nodes, _p(ntpn), _p(itin), _p(stage_base), _p(stage_pos))
    _ok("orc_hier_stage_pos", rc)
    return stage_base, stage_pos


def hier_dispatch(x, lay: dict, note: dict, stage_base, stage_pos, R: int, num_nodes: int):
    xb = _np(x, np.uint16)
    _, T, H = xb.shape
    n_stage = int(stage_base[R])
    staging = np.zeros((n_stage, H), np.uint16)
    ssr = np.empty(n_stage, np.int32)
    ssi = np.empty(n_stage, np.int32)
    rc = lib().orc_hier_stage_a(R, T, H, num_nodes, _p(xb), _p(_np(stage_pos, np.int32)), _p(staging),
                                _p(ssr), _p(ssi))
    _ok("orc_hier_stage_a", rc)
    n = int(note["rank_base"][R])
    recv_x = np.zeros((n, H), np.uint16)
    rc = lib().orc_hier_stage_b(R, T, H, num_nodes, n_stage, _p(_np(stage_base, np.int32)), _p(staging),
                                _p(ssr), _p(ssi), _p(_np(lay["is_token_in_rank"], np.uint8)),
                                _p(_np(note["send_pos"], np.int32)), _p(_np(note["rank_base"], np.int32)),
                                _p(recv_x))
    _ok("orc_hier_stage_b", rc)
    return dict(staging=staging, stage_src_rank=ssr, stage_src_idx=ssi, recv_x=recv_x)


# ---------------------------------------------------------------------------
# whole normal-mode chain (used by the parity tests and the CPU baseline)
# ---------------------------------------------------------------------------

def run_normal(x, topk_idx, topk_weights, R: int, E: int, C: int, combine_mode: str = "ord32"):
    idx = _np(topk_idx, np.int64)
    T = idx.shape[1]
    lay = layout(idx, R, E)
    note = notify(lay, R, E, T, C)
    disp = dispatch(x, idx, topk_weights, note, R, E)
    perm = permute(idx, disp["recv_x"], note, R, E)
    out = combine(perm["permuted_x"], perm["perm_pos"], idx, topk_weights, R, E, combine_mode)
    return dict(layout=lay, notify=note, dispatch=disp, permute=perm, out=out)
