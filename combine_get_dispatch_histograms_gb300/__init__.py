"""GB300-native MoE expert-parallel dispatch / combine.

A thin Python binding over the C ABI of libep_gb300.so (include/ep.h): it
only allocates device tensors with PyTorch, passes their pointers and the
current CUDA stream, and raises on a non-OK status.  Every step of the path
runs in the library's CUDA kernels; there is no CPU fallback, and using the
binding without the built library (or without a GPU) raises.

    ctx = Context(num_ranks=8, num_experts=256, num_topk=8, num_tokens=4096, hidden=7168)
    layout = ctx.get_dispatch_layout(topk_idx)
    handle = ctx.notify_dispatch(topk_idx, layout)          # the one host sync
    recv = ctx.dispatch(x, topk_idx, topk_weights, handle)
    perm = ctx.permute(handle, recv)
    out = ctx.combine(handle, expert_out, topk_idx, topk_weights)

    ll = LLBuffer(num_ranks=16, num_experts=256, num_topk=8, num_tokens=128, hidden=7168, cap=128)
    pk = ll.dispatch(x, topk_idx)                            # FP8, no host sync
    out = ll.combine(y_ll, topk_idx, topk_weights, pk)
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import EpConfig, EpDispatchHandle, EpError, check

__all__ = ["Context", "LLBuffer", "EpError", "load_library", "ll_size_hint", "ll_message_bytes"]


def load_library():
    return _lib.load()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    """cudaStream_t of `stream`, or of torch's current stream on the current device."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors passed to the CUDA path must be on a CUDA device")


def ll_message_bytes(hidden: int) -> int:
    return int(_lib.load().ep_ll_message_bytes(hidden))


def ll_size_hint(num_max_dispatch_tokens_per_rank: int, hidden: int, num_ranks: int, num_experts: int) -> int:
    return int(_lib.load().ep_ll_size_hint(num_max_dispatch_tokens_per_rank, hidden, num_ranks, num_experts))


class Handle(dict):
    """Device arrays of the dispatch handle plus the host counts of notify."""

    _cs = None
    _hrecv = None  # host arrays the waiting notify writes (owned by this handle)
    _hexp = None
    synced = False

    @property
    def host_num_recv_tokens(self):
        """[R] rows each receiver gets (waiting notify only, else None)."""
        return self._hrecv[:] if self.synced and self._hrecv is not None else None

    @property
    def host_num_recv_per_expert(self):
        """[R*L] pairs of each (receiver, local expert) (waiting notify only, else None)."""
        return self._hexp[:] if self.synced and self._hexp is not None else None

    def __setitem__(self, key, value):
        self._cs = None
        super().__setitem__(key, value)

    def c_struct(self) -> EpDispatchHandle:
        if self._cs is None:
            h = EpDispatchHandle()
            for name, _ in EpDispatchHandle._fields_:
                t = self.get(name)
                setattr(h, name, None if t is None else t.data_ptr())
            self._cs = h
        return self._cs


class Context:
    """Normal (high-throughput) mode over R virtual ranks on one GPU."""

    def __init__(self, num_ranks: int, num_experts: int, num_topk: int, num_tokens: int, hidden: int,
                 num_channels: int = 8, num_nodes: int = 1, device=None, expert_alignment: int = 1):
        if not torch.cuda.is_available():
            raise RuntimeError("the EP library needs a CUDA GPU")
        self.lib = _lib.load()
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.R, self.E, self.K, self.T, self.H = num_ranks, num_experts, num_topk, num_tokens, hidden
        self.C, self.N = num_channels, num_nodes
        self.L = num_experts // num_ranks
        self.cfg = EpConfig(num_ranks, num_experts, num_topk, num_tokens, hidden, num_channels, num_nodes)
        self._ctx = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            check("ep_ctx_create", self.lib.ep_ctx_create(ctypes.byref(self.cfg), ctypes.byref(self._ctx)))
        self.expert_alignment = 1
        if expert_alignment != 1:
            self.set_expert_alignment(expert_alignment)
        self._host_recv = (ctypes.c_int32 * num_ranks)()
        self._host_exp = (ctypes.c_int32 * num_experts)()
        self._host_tot = (ctypes.c_int32 * 3)()

    def close(self):
        if self._ctx:
            self.lib.ep_ctx_destroy(self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _i32(self, *shape):
        return torch.empty(*shape, dtype=torch.int32, device=self.device)

    @property
    def last_launches(self) -> int:
        return int(self.lib.ep_ctx_last_launches(self._ctx))

    def set_wait_timeout_us(self, us: int):
        check("ep_ctx_set_wait_timeout_us", self.lib.ep_ctx_set_wait_timeout_us(self._ctx, int(us)))

    def check(self, stream=None):
        check("ep_ctx_check", self.lib.ep_ctx_check(self._ctx, _stream(stream)))

    def set_expert_alignment(self, alignment: int):
        """Round every permuted expert block up to a multiple of `alignment` rows
        (from the next notify on); padding rows are left unwritten."""
        check("ep_ctx_set_expert_alignment", self.lib.ep_ctx_set_expert_alignment(self._ctx, int(alignment)))
        self.expert_alignment = int(alignment)

    # ---- layout ----------------------------------------------------------------
    def get_dispatch_layout(self, topk_idx: torch.Tensor, nodes: Optional[bool] = None, stream=None, out=None):
        _require_cuda(topk_idx)
        assert topk_idx.dtype == torch.int64 and topk_idx.is_contiguous()
        nodes = self.N > 1 if nodes is None else nodes
        R, E, T, N = self.R, self.E, self.T, self.N
        o = out if out is not None else dict(
            num_tokens_per_expert=self._i32(R, E),
            num_tokens_per_rank=self._i32(R, R),
            is_token_in_rank=torch.empty(R, T, R, dtype=torch.uint8, device=self.device),
        )
        if nodes and "num_tokens_per_node" not in o:
            o["num_tokens_per_node"] = self._i32(R, N)
            o["is_token_in_node"] = torch.empty(R, T, N, dtype=torch.uint8, device=self.device)
        check("ep_get_dispatch_layout", self.lib.ep_get_dispatch_layout(
            self._ctx, _ptr(topk_idx), _ptr(o["num_tokens_per_expert"]), _ptr(o["num_tokens_per_rank"]),
            _ptr(o["is_token_in_rank"]), _ptr(o.get("num_tokens_per_node") if nodes else None),
            _ptr(o.get("is_token_in_node") if nodes else None), _stream(stream)))
        return o

    # ---- notify ----------------------------------------------------------------
    def alloc_handle(self) -> Handle:
        R, T, K, L, C, N = self.R, self.T, self.K, self.L, self.C, self.N
        h = Handle(
            recv_count=self._i32(R, R), recv_offsets=self._i32(R, R), num_recv_tokens=self._i32(R),
            rank_base=self._i32(R + 1), num_recv_per_expert=self._i32(R, L), expert_offsets=self._i32(R, L),
            perm_rank_base=self._i32(R + 1), channel_prefix_matrix=self._i32(R, R, C),
            send_pos=self._i32(R, T, R), perm_pos=self._i32(R, T, K))
        if N > 1:
            h["stage_base"] = self._i32(R + 1)
            h["stage_pos"] = self._i32(R, T, N)
        return h

    @property
    def max_rows(self) -> tuple:
        """Worst-case (received, permuted, staged) row counts: buffers of these
        sizes never overflow, whatever the routing."""
        R, T, K, N = self.R, self.T, self.K, self.N
        pad = self.E * (self.expert_alignment - 1)
        return R * T * min(K, R), R * T * K + pad, (R * T * min(K, N) if N > 1 else 0)

    def notify_dispatch(self, topk_idx: torch.Tensor, layout: dict, stream=None, handle: Optional[Handle] = None,
                        wait: bool = True) -> Handle:
        """wait=False: no host synchronisation (graph-capturable).  The row
        totals then stay on the device (handle["rank_base"][R], ["perm_rank_base"][R],
        ["stage_base"][R]) and the handle's num_*_rows are the worst-case bounds."""
        return self._notify("ep_notify_dispatch", topk_idx, layout, stream, handle, wait)

    def layout_notify(self, topk_idx: torch.Tensor, stream=None, handle: Optional[Handle] = None,
                      out: Optional[dict] = None, wait: bool = True):
        """get_dispatch_layout and notify_dispatch in two launches instead of
        three; returns (layout dict, handle), the same as the two calls."""
        _require_cuda(topk_idx)
        R, E, T, N = self.R, self.E, self.T, self.N
        lay = out if out is not None else dict(
            num_tokens_per_expert=self._i32(R, E), num_tokens_per_rank=self._i32(R, R),
            is_token_in_rank=torch.empty(R, T, R, dtype=torch.uint8, device=self.device))
        if N > 1 and "num_tokens_per_node" not in lay:
            lay["num_tokens_per_node"] = self._i32(R, N)
            lay["is_token_in_node"] = torch.empty(R, T, N, dtype=torch.uint8, device=self.device)
        return lay, self._notify("ep_layout_notify", topk_idx, lay, stream, handle, wait)

    def _notify(self, fn: str, topk_idx, layout: dict, stream, handle: Optional[Handle], wait: bool) -> Handle:
        _require_cuda(topk_idx)
        h = handle if handle is not None else self.alloc_handle()
        cs = h.c_struct()
        if wait:
            if h._hrecv is None:  # the handle's own host arrays: no copy after the wait
                h._hrecv = (ctypes.c_int32 * self.R)()
                h._hexp = (ctypes.c_int32 * self.E)()
            host_recv, host_exp, host_tot = h._hrecv, h._hexp, self._host_tot
        else:
            host_recv = host_exp = host_tot = None
        nodes = self.N > 1 or fn == "ep_notify_dispatch"
        check(fn, getattr(self.lib, fn)(
            self._ctx, _ptr(topk_idx), _ptr(layout["num_tokens_per_expert"]), _ptr(layout["num_tokens_per_rank"]),
            _ptr(layout["is_token_in_rank"]), _ptr(layout.get("num_tokens_per_node") if nodes else None),
            _ptr(layout.get("is_token_in_node") if nodes else None), ctypes.byref(cs), host_recv, host_exp, host_tot,
            _stream(stream)))
        h.synced = wait
        if wait:
            h.num_recv_rows, h.num_perm_rows, h.num_stage_rows = host_tot
        else:
            h.num_recv_rows, h.num_perm_rows, h.num_stage_rows = self.max_rows
        return h

    # ---- dispatch / permute ----------------------------------------------------
    @staticmethod
    def _recv_rows(handle: Handle, recv_rows: torch.Tensor) -> int:
        # rows permute may read: the waited total, else the recv buffer's capacity
        return handle.num_recv_rows if getattr(handle, "synced", True) else recv_rows.shape[0]

    def alloc_recv(self, rows: int) -> dict:
        return dict(
            recv_x=torch.empty(rows, self.H, dtype=torch.bfloat16, device=self.device),
            recv_src_rank=self._i32(rows), recv_src_idx=self._i32(rows),
            recv_topk_idx=self._i32(rows, self.K),
            recv_topk_weights=torch.empty(rows, self.K, dtype=torch.float32, device=self.device))

    def dispatch(self, x, topk_idx, topk_weights, handle: Handle, stream=None, out=None) -> dict:
        _require_cuda(x, topk_idx, topk_weights)
        assert x.dtype == torch.bfloat16 and x.is_contiguous()
        o = out if out is not None else self.alloc_recv(handle.num_recv_rows)
        cs = handle.c_struct()
        check("ep_dispatch", self.lib.ep_dispatch(
            self._ctx, _ptr(x), _ptr(topk_idx), _ptr(topk_weights), ctypes.byref(cs), _ptr(o["recv_x"]),
            _ptr(o["recv_src_rank"]), _ptr(o["recv_src_idx"]), _ptr(o["recv_topk_idx"]),
            _ptr(o["recv_topk_weights"]), o["recv_x"].shape[0], _stream(stream)))
        return o

    def permute(self, handle: Handle, recv: dict, stream=None, out=None) -> dict:
        P = handle.num_perm_rows
        o = out if out is not None else dict(
            permuted_x=torch.empty(P, self.H, dtype=torch.bfloat16, device=self.device),
            perm_src_row=self._i32(P))
        cs = handle.c_struct()
        check("ep_permute", self.lib.ep_permute(
            self._ctx, ctypes.byref(cs), _ptr(recv["recv_x"]), _ptr(recv["recv_src_rank"]),
            _ptr(recv["recv_src_idx"]), _ptr(recv["recv_topk_idx"]), self._recv_rows(handle, recv["recv_x"]),
            _ptr(o["permuted_x"]), _ptr(o["perm_src_row"]), o["permuted_x"].shape[0], _stream(stream)))
        return o

    def dispatch_permuted(self, x, topk_idx, topk_weights, handle: Handle, stream=None, out=None) -> dict:
        """Fused dispatch: tokens straight into the expert-major layout."""
        _require_cuda(x, topk_idx, topk_weights)
        P = handle.num_perm_rows
        o = out if out is not None else dict(
            permuted_x=torch.empty(P, self.H, dtype=torch.bfloat16, device=self.device),
            perm_src_token=self._i32(P), perm_weight=torch.empty(P, dtype=torch.float32, device=self.device))
        cs = handle.c_struct()
        check("ep_dispatch_permuted", self.lib.ep_dispatch_permuted(
            self._ctx, _ptr(x), _ptr(topk_idx), _ptr(topk_weights), ctypes.byref(cs), _ptr(o["permuted_x"]),
            _ptr(o["perm_src_token"]), _ptr(o.get("perm_weight")), o["permuted_x"].shape[0], _stream(stream)))
        return o

    # ---- FP8 rows ----------------------------------------------------------------
    @property
    def fp8_row_bytes(self) -> int:
        return int(self.lib.ep_fp8_row_bytes(self.H))

    def quantize_fp8(self, x, stream=None, out=None):
        """Every token once into an FP8 row (H e4m3 codes, H/128 fp32 scales)."""
        _require_cuda(x)
        o = out if out is not None else torch.empty(self.R * self.T, self.fp8_row_bytes, dtype=torch.uint8,
                                                    device=self.device)
        check("ep_quantize_fp8", self.lib.ep_quantize_fp8(self._ctx, _ptr(x), _ptr(o), _stream(stream)))
        return o

    def dispatch_fp8(self, xq, topk_idx, topk_weights, handle: Handle, stream=None, out=None) -> dict:
        rows = handle.num_recv_rows
        o = out if out is not None else dict(
            recv_xq=torch.empty(rows, self.fp8_row_bytes, dtype=torch.uint8, device=self.device),
            recv_src_rank=self._i32(rows), recv_src_idx=self._i32(rows), recv_topk_idx=self._i32(rows, self.K),
            recv_topk_weights=torch.empty(rows, self.K, dtype=torch.float32, device=self.device))
        cs = handle.c_struct()
        check("ep_dispatch_fp8", self.lib.ep_dispatch_fp8(
            self._ctx, _ptr(xq), _ptr(topk_idx), _ptr(topk_weights), ctypes.byref(cs), _ptr(o["recv_xq"]),
            _ptr(o["recv_src_rank"]), _ptr(o["recv_src_idx"]), _ptr(o["recv_topk_idx"]),
            _ptr(o["recv_topk_weights"]), o["recv_xq"].shape[0], _stream(stream)))
        return o

    def permute_fp8(self, handle: Handle, recv: dict, stream=None, out=None) -> dict:
        P = handle.num_perm_rows
        o = out if out is not None else dict(
            permuted_xq=torch.empty(P, self.fp8_row_bytes, dtype=torch.uint8, device=self.device),
            perm_src_row=self._i32(P))
        cs = handle.c_struct()
        check("ep_permute_fp8", self.lib.ep_permute_fp8(
            self._ctx, ctypes.byref(cs), _ptr(recv["recv_xq"]), _ptr(recv["recv_src_rank"]),
            _ptr(recv["recv_src_idx"]), _ptr(recv["recv_topk_idx"]), self._recv_rows(handle, recv["recv_xq"]),
            _ptr(o["permuted_xq"]), _ptr(o["perm_src_row"]), o["permuted_xq"].shape[0], _stream(stream)))
        return o

    def dispatch_permuted_fp8(self, xq, topk_idx, topk_weights, handle: Handle, stream=None, out=None) -> dict:
        P = handle.num_perm_rows
        o = out if out is not None else dict(
            permuted_xq=torch.empty(P, self.fp8_row_bytes, dtype=torch.uint8, device=self.device),
            perm_src_token=self._i32(P), perm_weight=torch.empty(P, dtype=torch.float32, device=self.device))
        cs = handle.c_struct()
        check("ep_dispatch_permuted_fp8", self.lib.ep_dispatch_permuted_fp8(
            self._ctx, _ptr(xq), _ptr(topk_idx), _ptr(topk_weights), ctypes.byref(cs), _ptr(o["permuted_xq"]),
            _ptr(o["perm_src_token"]), _ptr(o.get("perm_weight")), o["permuted_xq"].shape[0], _stream(stream)))
        return o

    def dispatch_quant(self, x, topk_idx, topk_weights, handle: Handle, stream=None, out=None) -> dict:
        """Quantise the bf16 tokens and scatter the FP8 rows to the receive
        layout in one pass (quantize_fp8 + dispatch_fp8 fused)."""
        _require_cuda(x, topk_idx, topk_weights)
        rows = handle.num_recv_rows
        o = out if out is not None else dict(
            recv_xq=torch.empty(rows, self.fp8_row_bytes, dtype=torch.uint8, device=self.device),
            recv_src_rank=self._i32(rows), recv_src_idx=self._i32(rows), recv_topk_idx=self._i32(rows, self.K),
            recv_topk_weights=torch.empty(rows, self.K, dtype=torch.float32, device=self.device))
        cs = handle.c_struct()
        check("ep_dispatch_quant", self.lib.ep_dispatch_quant(
            self._ctx, _ptr(x), _ptr(topk_idx), _ptr(topk_weights), ctypes.byref(cs), _ptr(o["recv_xq"]),
            _ptr(o["recv_src_rank"]), _ptr(o["recv_src_idx"]), _ptr(o["recv_topk_idx"]),
            _ptr(o["recv_topk_weights"]), o["recv_xq"].shape[0], _stream(stream)))
        return o

    def dispatch_permuted_quant(self, x, topk_idx, topk_weights, handle: Handle, stream=None, out=None) -> dict:
        """Quantise the bf16 tokens and dispatch the FP8 rows into the permuted
        layout in one pass (quantize_fp8 + dispatch_permuted_fp8 fused)."""
        _require_cuda(x, topk_idx, topk_weights)
        P = handle.num_perm_rows
        o = out if out is not None else dict(
            permuted_xq=torch.empty(P, self.fp8_row_bytes, dtype=torch.uint8, device=self.device),
            perm_src_token=self._i32(P), perm_weight=torch.empty(P, dtype=torch.float32, device=self.device))
        cs = handle.c_struct()
        check("ep_dispatch_permuted_quant", self.lib.ep_dispatch_permuted_quant(
            self._ctx, _ptr(x), _ptr(topk_idx), _ptr(topk_weights), ctypes.byref(cs), _ptr(o["permuted_xq"]),
            _ptr(o["perm_src_token"]), _ptr(o.get("perm_weight")), o["permuted_xq"].shape[0], _stream(stream)))
        return o

    # ---- combine ---------------------------------------------------------------
    def combine(self, handle: Handle, expert_out, topk_idx, topk_weights, stream=None, out=None, hier=False):
        _require_cuda(expert_out, topk_idx, topk_weights)
        o = out if out is not None else torch.empty(self.R, self.T, self.H, dtype=torch.bfloat16, device=self.device)
        cs = handle.c_struct()
        fn = self.lib.ep_combine_hier if hier else self.lib.ep_combine
        check("ep_combine_hier" if hier else "ep_combine", fn(
            self._ctx, ctypes.byref(cs), _ptr(expert_out), expert_out.shape[0], _ptr(topk_idx), _ptr(topk_weights),
            _ptr(o), _stream(stream)))
        return o

    def combine_hier(self, handle, expert_out, topk_idx, topk_weights, stream=None, out=None):
        return self.combine(handle, expert_out, topk_idx, topk_weights, stream=stream, out=out, hier=True)

    # ---- hierarchical dispatch -------------------------------------------------
    def dispatch_hier(self, x, topk_idx, topk_weights, handle: Handle, stream=None, out=None, staging=None) -> dict:
        _require_cuda(x, topk_idx, topk_weights)
        o = out if out is not None else self.alloc_recv(handle.num_recv_rows)
        S = handle.num_stage_rows
        st = staging if staging is not None else dict(
            staging=torch.empty(S, self.H, dtype=torch.bfloat16, device=self.device),
            stage_src_rank=self._i32(S), stage_src_idx=self._i32(S))
        cs = handle.c_struct()
        check("ep_dispatch_hier", self.lib.ep_dispatch_hier(
            self._ctx, _ptr(x), _ptr(topk_idx), _ptr(topk_weights), ctypes.byref(cs), _ptr(st["staging"]),
            _ptr(st["stage_src_rank"]), _ptr(st["stage_src_idx"]), st["staging"].shape[0], _ptr(o["recv_x"]),
            _ptr(o["recv_src_rank"]), _ptr(o["recv_src_idx"]), _ptr(o["recv_topk_idx"]),
            _ptr(o["recv_topk_weights"]), o["recv_x"].shape[0], _stream(stream)))
        o.update(st)
        return o


class LLBuffer:
    """Low-latency mode: fixed (expert, source) regions, FP8 dispatch, BF16 combine."""

    def __init__(self, num_ranks: int, num_experts: int, num_topk: int, num_tokens: int, hidden: int, cap: int,
                 device=None):
        if not torch.cuda.is_available():
            raise RuntimeError("the EP library needs a CUDA GPU")
        self.lib = _lib.load()
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.R, self.E, self.K, self.T, self.H, self.cap = num_ranks, num_experts, num_topk, num_tokens, hidden, cap
        self.L = num_experts // num_ranks
        self.cfg = EpConfig(num_ranks, num_experts, num_topk, num_tokens, hidden, 1, 1)
        self._buf = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            check("ep_ll_buffer_create", self.lib.ep_ll_buffer_create(ctypes.byref(self.cfg), cap, ctypes.byref(self._buf)))

    def close(self):
        if self._buf:
            self.lib.ep_ll_buffer_destroy(self._buf)
            self._buf = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_wait_timeout_us(self, us: int):
        check("ep_ll_set_wait_timeout_us", self.lib.ep_ll_set_wait_timeout_us(self._buf, int(us)))

    def check(self, stream=None):
        check("ep_ll_check", self.lib.ep_ll_check(self._buf, _stream(stream)))

    def trace_waits(self, wait_ns: Optional[torch.Tensor]):
        """From the next receive on, write each (expert, source) signal wait (ns)
        into wait_ns [E][R] int64 on the device; None stops the trace."""
        if wait_ns is not None:
            assert wait_ns.is_cuda and wait_ns.dtype == torch.int64 and wait_ns.numel() == self.E * self.R
        self._trace = wait_ns  # kept alive while the library holds its address
        check("ep_ll_set_wait_trace", self.lib.ep_ll_set_wait_trace(self._buf, _ptr(wait_ns)))

    def count_slots(self, which: int) -> int:
        return int(self.lib.ep_ll_count_slots(self._buf, which) or 0)

    @property
    def current_buffer(self) -> int:
        return int(self.lib.ep_ll_current_buffer(self._buf))

    def alloc_packed(self) -> dict:
        R, L, cap, H = self.R, self.L, self.cap, self.H
        i32 = lambda *s: torch.empty(*s, dtype=torch.int32, device=self.device)
        return dict(
            packed_x=torch.empty(R, L, R * cap, H, dtype=torch.uint8, device=self.device),
            packed_scales=torch.empty(R, L, R * cap, H // 128, dtype=torch.float32, device=self.device),
            packed_src_info=i32(R, L, R * cap, 2), packed_recv_count=i32(R, L), layout_range=i32(R, L, R, 2),
            slot=i32(self.R, self.T, self.K))

    def send(self, x, topk_idx, t0: int = 0, n: Optional[int] = None, stream=None, out=None) -> dict:
        _require_cuda(x, topk_idx)
        n = self.T - t0 if n is None else n
        o = out if out is not None else self.alloc_packed()
        check("ep_ll_send", self.lib.ep_ll_send(self._buf, _ptr(x), _ptr(topk_idx), t0, n, _ptr(o["slot"]),
                                                 _stream(stream)))
        return o

    def recv(self, out: dict, stream=None) -> dict:
        check("ep_ll_recv", self.lib.ep_ll_recv(self._buf, _ptr(out["packed_x"]), _ptr(out["packed_scales"]),
                                                 _ptr(out["packed_src_info"]), _ptr(out["packed_recv_count"]),
                                                 _ptr(out["layout_range"]), _stream(stream)))
        return out

    def dispatch(self, x, topk_idx, t0: int = 0, n: Optional[int] = None, stream=None, out=None) -> dict:
        _require_cuda(x, topk_idx)
        n = self.T - t0 if n is None else n
        o = out if out is not None else self.alloc_packed()
        check("ep_ll_dispatch", self.lib.ep_ll_dispatch(
            self._buf, _ptr(x), _ptr(topk_idx), t0, n, _ptr(o["packed_x"]), _ptr(o["packed_scales"]),
            _ptr(o["packed_src_info"]), _ptr(o["packed_recv_count"]), _ptr(o["layout_range"]), _ptr(o["slot"]),
            _stream(stream)))
        return o

    def combine(self, y_ll, topk_idx, topk_weights, packed: dict, t0: int = 0, n: Optional[int] = None,
                stream=None, out=None):
        _require_cuda(y_ll, topk_idx, topk_weights)
        n = self.T - t0 if n is None else n
        o = out if out is not None else torch.zeros(self.R, self.T, self.H, dtype=torch.bfloat16, device=self.device)
        check("ep_ll_combine", self.lib.ep_ll_combine(
            self._buf, _ptr(y_ll), _ptr(topk_idx), _ptr(topk_weights), _ptr(packed["slot"]),
            _ptr(packed["layout_range"]), t0, n, _ptr(o), _stream(stream)))
        return o
