"""Python binding of libmoe_route.so (GB300 MoE token routing).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are PyTorch CUDA tensors (device memory and streams come from
PyTorch); they are checked for device, contiguity and size before their raw
pointers are handed to the C ABI declared in ``include/moe_route.h``.

The library is built in-tree by ``combine_moe_route_topk_gb300._build``
(``__graft_entry__.build()``); importing an op without it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import workloads  # noqa: F401  (re-exported for convenience)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_route.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_CAPACITY = -4
MOE_ERR_TIMEOUT = -5

MOE_BF16, MOE_F32, MOE_FP8E4M3_BLK128 = 0, 1, 2
MOE_SOFTMAX, MOE_SIGMOID = 0, 1
MOE_BIAS_SELECT_ONLY = 0x10  # OR into score_fn: the bias enters the selection key only

STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
                -3: "MOE_ERR_CUDA", -4: "MOE_ERR_CAPACITY", -5: "MOE_ERR_TIMEOUT"}

_TORCH_DTYPE = {MOE_BF16: torch.bfloat16, MOE_F32: torch.float32, MOE_FP8E4M3_BLK128: torch.uint8}


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class MoeDims(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int32), ("T", ctypes.c_int32), ("E", ctypes.c_int32),
                ("R", ctypes.c_int32), ("H", ctypes.c_int32), ("x_dtype", ctypes.c_int32),
                ("y_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cap_rows", ctypes.c_int64)]


_SIZE_FIELDS = ["bound_rows", "cap_rows", "total_pairs", "logits_bytes", "topk_idx_bytes",
                "topk_w_bytes", "pos_bytes", "expert_counts_bytes", "expert_offsets_bytes",
                "rank_counts_bytes", "rank_offsets_bytes", "send_counts_bytes", "x_bytes",
                "x_scales_bytes", "packed_x_bytes", "packed_scales_bytes", "packed_src_bytes",
                "y_bytes", "out_bytes", "status_bytes", "partial_slots", "partial_bytes",
                "slot_rank_bytes", "fused_workspace_bytes"]


class MoeSizes(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int64) for f in _SIZE_FIELDS]

    def as_dict(self) -> dict:
        return {f: int(getattr(self, f)) for f in _SIZE_FIELDS}


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe_route.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                    f"g.build()'` (needs nvcc); there is no fallback implementation")
            L = ctypes.CDLL(LIB_PATH)
            P, i32 = ctypes.c_void_p, ctypes.c_int
            D = ctypes.POINTER(MoeDims)
            L.moe_buffer_sizes.argtypes = [D, ctypes.POINTER(MoeSizes)]
            L.moe_route_topk.argtypes = [D, P, P, i32, i32, P, P, P]
            L.moe_dispatch_count.argtypes = [D, P, P, P, P, P, P, P, P, P]
            L.moe_dispatch_pack.argtypes = [D, P, P, P, P, P, P, P]
            L.moe_combine.argtypes = [D, P, P, P, P, P]
            L.moe_dispatch_pack_quant.argtypes = [D, P, P, P, P, P, P]
            L.moe_dispatch_pack_rank.argtypes = [D, i32, P, P, P, P, P, P, P]
            L.moe_dispatch_fused.argtypes = [D, P, P, i32, i32, P, P, P, P, P, P, P, P, P, P, P,
                                             P, P, P, P, P]
            L.moe_dispatch_fused_static.argtypes = [D, P, P, i32, i32, P, P, P, P, P, P, P, P, P,
                                                    P, P, P, P, P, P]
            L.moe_combine_rank.argtypes = [D, i32, P, P, P, P, P]
            L.moe_combine_partials.argtypes = [D, P, P, P, P, P, P]
            L.moe_combine_reduce_partials.argtypes = [D, P, P, P, P]
            L.moe_read_status.argtypes = [P, P]
            L.moe_take_device_error.argtypes = [P]
            L.moe_selftest_bounded_wait.argtypes = [P, ctypes.c_int64, P]
            L.moe_last_error.restype = ctypes.c_char_p
            L.moe_last_error.argtypes = []
            L.moe_version.restype = i32
            for fn in ("moe_buffer_sizes", "moe_route_topk", "moe_dispatch_count",
                       "moe_dispatch_pack", "moe_dispatch_pack_quant", "moe_dispatch_pack_rank",
                       "moe_dispatch_fused", "moe_dispatch_fused_static",
                       "moe_combine", "moe_combine_rank", "moe_combine_partials",
                       "moe_combine_reduce_partials", "moe_read_status",
                       "moe_take_device_error", "moe_selftest_bounded_wait"):
                getattr(L, fn).restype = i32
            _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, lib().moe_last_error().decode())


def make_dims(N, T, E, R, H, x_dtype=MOE_BF16, y_dtype=MOE_BF16, cap_rows=0) -> MoeDims:
    return MoeDims(N, T, E, R, H, x_dtype, y_dtype, 0, cap_rows)


def dims_of(w) -> MoeDims:
    """MoeDims of a ``workloads.Workload``."""
    return make_dims(w.N, w.T, w.E, w.R, w.H, w.x_dtype, w.y_dtype, w.cap_rows)


_sizes_cache: dict = {}


def buffer_sizes(dims: MoeDims) -> dict:
    """Buffer sizes for ``dims`` (memoised: the query is pure host arithmetic)."""
    key = bytes(dims)
    hit = _sizes_cache.get(key)
    if hit is not None:
        return hit
    s = MoeSizes()
    _check(lib().moe_buffer_sizes(ctypes.byref(dims), ctypes.byref(s)))
    d = s.as_dict()
    if len(_sizes_cache) < 256:
        _sizes_cache[key] = d
    return d


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor | None, nbytes: int, name: str, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not the current device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes, needs {nbytes}")
    return ctypes.c_void_p(t.data_ptr())


def route_topk(dims: MoeDims, logits, bias, score_fn, renormalize, topk_idx, topk_w, stream=None):
    s = buffer_sizes(dims)
    _check(lib().moe_route_topk(
        ctypes.byref(dims), _ptr(logits, s["logits_bytes"], "logits", torch.float32),
        _ptr(bias, dims.E * 4, "bias", torch.float32, optional=True), int(score_fn),
        int(bool(renormalize)), _ptr(topk_idx, s["topk_idx_bytes"], "topk_idx", torch.int32),
        _ptr(topk_w, s["topk_w_bytes"], "topk_w", torch.float32), _stream(stream)))


def dispatch_count(dims: MoeDims, topk_idx, expert_counts, expert_offsets, rank_counts,
                   rank_offsets, send_counts, pos, status, stream=None):
    s = buffer_sizes(dims)
    i32 = torch.int32
    _check(lib().moe_dispatch_count(
        ctypes.byref(dims), _ptr(topk_idx, s["topk_idx_bytes"], "topk_idx", i32),
        _ptr(expert_counts, s["expert_counts_bytes"], "expert_counts", i32),
        _ptr(expert_offsets, s["expert_offsets_bytes"], "expert_offsets", i32),
        _ptr(rank_counts, s["rank_counts_bytes"], "rank_counts", i32),
        _ptr(rank_offsets, s["rank_offsets_bytes"], "rank_offsets", i32),
        _ptr(send_counts, s["send_counts_bytes"], "send_counts", i32),
        _ptr(pos, s["pos_bytes"], "pos", i32), _ptr(status, 4, "status", i32), _stream(stream)))


def dispatch_pack(dims: MoeDims, x, x_scales, pos, packed_x, packed_scales, packed_src,
                  stream=None):
    s = buffer_sizes(dims)
    fp8 = dims.x_dtype == MOE_FP8E4M3_BLK128
    _check(lib().moe_dispatch_pack(
        ctypes.byref(dims), _ptr(x, s["x_bytes"], "x", _TORCH_DTYPE[dims.x_dtype]),
        _ptr(x_scales, s["x_scales_bytes"], "x_scales", torch.float32, optional=not fp8),
        _ptr(pos, s["pos_bytes"], "pos", torch.int32),
        _ptr(packed_x, s["packed_x_bytes"], "packed_x", _TORCH_DTYPE[dims.x_dtype]),
        _ptr(packed_scales, s["packed_scales_bytes"], "packed_scales", torch.float32,
             optional=not fp8),
        _ptr(packed_src, s["packed_src_bytes"], "packed_src", torch.int32), _stream(stream)))


def dispatch_fused(dims: MoeDims, logits, bias, score_fn, renormalize, x, x_scales, topk_idx,
                   topk_w, expert_counts, expert_offsets, rank_counts, rank_offsets, send_counts,
                   pos, status, packed_x, packed_scales, packed_src, workspace, stream=None):
    """Route + count + pack in one launch (decode batches)."""
    s = buffer_sizes(dims)
    i32, f32 = torch.int32, torch.float32
    fp8 = dims.x_dtype == MOE_FP8E4M3_BLK128
    _check(lib().moe_dispatch_fused(
        ctypes.byref(dims), _ptr(logits, s["logits_bytes"], "logits", f32),
        _ptr(bias, dims.E * 4, "bias", f32, optional=True), int(score_fn), int(bool(renormalize)),
        _ptr(x, s["x_bytes"], "x", _TORCH_DTYPE[dims.x_dtype]),
        _ptr(x_scales, s["x_scales_bytes"], "x_scales", f32, optional=not fp8),
        _ptr(topk_idx, s["topk_idx_bytes"], "topk_idx", i32),
        _ptr(topk_w, s["topk_w_bytes"], "topk_w", f32),
        _ptr(expert_counts, s["expert_counts_bytes"], "expert_counts", i32),
        _ptr(expert_offsets, s["expert_offsets_bytes"], "expert_offsets", i32),
        _ptr(rank_counts, s["rank_counts_bytes"], "rank_counts", i32),
        _ptr(rank_offsets, s["rank_offsets_bytes"], "rank_offsets", i32),
        _ptr(send_counts, s["send_counts_bytes"], "send_counts", i32),
        _ptr(pos, s["pos_bytes"], "pos", i32), _ptr(status, 4, "status", i32),
        _ptr(packed_x, s["packed_x_bytes"], "packed_x", _TORCH_DTYPE[dims.x_dtype]),
        _ptr(packed_scales, s["packed_scales_bytes"], "packed_scales", f32, optional=not fp8),
        _ptr(packed_src, s["packed_src_bytes"], "packed_src", i32),
        _ptr(workspace, s["fused_workspace_bytes"], "workspace", optional=dims.N * dims.T == 0),
        _stream(stream)))


def dispatch_fused_static(dims: MoeDims, logits, bias, score_fn, renormalize, x, x_scales,
                          topk_idx, topk_w, expert_counts, expert_offsets, rank_counts,
                          rank_offsets, send_counts, pos, status, packed_x, packed_scales,
                          packed_src, stream=None):
    """moe_dispatch_fused with the library's own static scratch: nothing is
    allocated by the call (for callers that cannot allocate device memory
    when they dispatch).  Calls that overlap on the GPU race on the scratch."""
    s = buffer_sizes(dims)
    i32, f32 = torch.int32, torch.float32
    fp8 = dims.x_dtype == MOE_FP8E4M3_BLK128
    _check(lib().moe_dispatch_fused_static(
        ctypes.byref(dims), _ptr(logits, s["logits_bytes"], "logits", f32),
        _ptr(bias, dims.E * 4, "bias", f32, optional=True), int(score_fn), int(bool(renormalize)),
        _ptr(x, s["x_bytes"], "x", _TORCH_DTYPE[dims.x_dtype]),
        _ptr(x_scales, s["x_scales_bytes"], "x_scales", f32, optional=not fp8),
        _ptr(topk_idx, s["topk_idx_bytes"], "topk_idx", i32),
        _ptr(topk_w, s["topk_w_bytes"], "topk_w", f32),
        _ptr(expert_counts, s["expert_counts_bytes"], "expert_counts", i32),
        _ptr(expert_offsets, s["expert_offsets_bytes"], "expert_offsets", i32),
        _ptr(rank_counts, s["rank_counts_bytes"], "rank_counts", i32),
        _ptr(rank_offsets, s["rank_offsets_bytes"], "rank_offsets", i32),
        _ptr(send_counts, s["send_counts_bytes"], "send_counts", i32),
        _ptr(pos, s["pos_bytes"], "pos", i32), _ptr(status, 4, "status", i32),
        _ptr(packed_x, s["packed_x_bytes"], "packed_x", _TORCH_DTYPE[dims.x_dtype]),
        _ptr(packed_scales, s["packed_scales_bytes"], "packed_scales", f32, optional=not fp8),
        _ptr(packed_src, s["packed_src_bytes"], "packed_src", i32), _stream(stream)))


def fp8_dims(dims: MoeDims) -> MoeDims:
    """The same problem with fp8 block-scaled rows (sizes of quantised buffers)."""
    return make_dims(dims.N, dims.T, dims.E, dims.R, dims.H, MOE_FP8E4M3_BLK128, dims.y_dtype,
                     dims.cap_rows)


def dispatch_pack_quant(dims: MoeDims, x, pos, packed_q, packed_scales, packed_src,
                        stream=None):
    """Pack bf16 rows as e4m3 codes + one f32 scale per 128 elements."""
    s = buffer_sizes(dims)
    q = buffer_sizes(fp8_dims(dims))
    _check(lib().moe_dispatch_pack_quant(
        ctypes.byref(dims), _ptr(x, s["x_bytes"], "x", torch.bfloat16),
        _ptr(pos, s["pos_bytes"], "pos", torch.int32),
        _ptr(packed_q, q["packed_x_bytes"], "packed_q", torch.uint8),
        _ptr(packed_scales, q["packed_scales_bytes"], "packed_scales", torch.float32),
        _ptr(packed_src, s["packed_src_bytes"], "packed_src", torch.int32), _stream(stream)))


def dispatch_fused_quant(dims: MoeDims, logits, bias, score_fn, renormalize, x, topk_idx, topk_w,
                         expert_counts, expert_offsets, rank_counts, rank_offsets, send_counts, pos,
                         status, packed_q, packed_scales, packed_src, workspace, stream=None):
    """Route + count + fp8-quantising pack in one call (decode batches; bf16 rows
    in, e4m3 codes + one f32 scale per 128 elements out)."""
    s = buffer_sizes(dims)
    q = buffer_sizes(fp8_dims(dims))
    i32, f32 = torch.int32, torch.float32
    _check(lib().moe_dispatch_fused_quant(
        ctypes.byref(dims), _ptr(logits, s["logits_bytes"], "logits", f32),
        _ptr(bias, dims.E * 4, "bias", f32, optional=True), int(score_fn), int(bool(renormalize)),
        _ptr(x, s["x_bytes"], "x", torch.bfloat16),
        _ptr(topk_idx, s["topk_idx_bytes"], "topk_idx", i32),
        _ptr(topk_w, s["topk_w_bytes"], "topk_w", f32),
        _ptr(expert_counts, s["expert_counts_bytes"], "expert_counts", i32),
        _ptr(expert_offsets, s["expert_offsets_bytes"], "expert_offsets", i32),
        _ptr(rank_counts, s["rank_counts_bytes"], "rank_counts", i32),
        _ptr(rank_offsets, s["rank_offsets_bytes"], "rank_offsets", i32),
        _ptr(send_counts, s["send_counts_bytes"], "send_counts", i32),
        _ptr(pos, s["pos_bytes"], "pos", i32), _ptr(status, 4, "status", i32),
        _ptr(packed_q, q["packed_x_bytes"], "packed_q", torch.uint8),
        _ptr(packed_scales, q["packed_scales_bytes"], "packed_scales", f32),
        _ptr(packed_src, s["packed_src_bytes"], "packed_src", i32),
        _ptr(workspace, s["fused_workspace_bytes"], "workspace", optional=dims.N * dims.T == 0),
        _stream(stream)))


def combine(dims: MoeDims, y, pos, topk_w, out, stream=None):
    s = buffer_sizes(dims)
    yt = _TORCH_DTYPE[dims.y_dtype]
    _check(lib().moe_combine(
        ctypes.byref(dims), _ptr(y, s["y_bytes"], "y", yt),
        _ptr(pos, s["pos_bytes"], "pos", torch.int32),
        _ptr(topk_w, s["topk_w_bytes"], "topk_w", torch.float32),
        _ptr(out, s["out_bytes"], "out", yt), _stream(stream)))


def dispatch_pack_rank(dims: MoeDims, rank: int, x, x_scales, pos, packed_x, packed_scales,
                       packed_src, stream=None):
    """moe_dispatch_pack restricted to the pairs routed to rank `rank`."""
    s = buffer_sizes(dims)
    fp8 = dims.x_dtype == MOE_FP8E4M3_BLK128
    _check(lib().moe_dispatch_pack_rank(
        ctypes.byref(dims), int(rank), _ptr(x, s["x_bytes"], "x", _TORCH_DTYPE[dims.x_dtype]),
        _ptr(x_scales, s["x_scales_bytes"], "x_scales", torch.float32, optional=not fp8),
        _ptr(pos, s["pos_bytes"], "pos", torch.int32),
        _ptr(packed_x, s["packed_x_bytes"], "packed_x", _TORCH_DTYPE[dims.x_dtype]),
        _ptr(packed_scales, s["packed_scales_bytes"], "packed_scales", torch.float32,
             optional=not fp8),
        _ptr(packed_src, s["packed_src_bytes"], "packed_src", torch.int32), _stream(stream)))


def combine_rank(dims: MoeDims, rank: int, y, pos, topk_w, out, stream=None):
    """Local accumulation of rank `rank` (dense [N*T][H])."""
    s = buffer_sizes(dims)
    yt = _TORCH_DTYPE[dims.y_dtype]
    _check(lib().moe_combine_rank(
        ctypes.byref(dims), int(rank), _ptr(y, s["y_bytes"], "y", yt),
        _ptr(pos, s["pos_bytes"], "pos", torch.int32),
        _ptr(topk_w, s["topk_w_bytes"], "topk_w", torch.float32),
        _ptr(out, s["out_bytes"], "out", yt), _stream(stream)))


def combine_partials(dims: MoeDims, y, pos, topk_w, partial, slot_rank, stream=None):
    """Per (token, destination rank) partial rows and their ranks."""
    s = buffer_sizes(dims)
    yt = _TORCH_DTYPE[dims.y_dtype]
    _check(lib().moe_combine_partials(
        ctypes.byref(dims), _ptr(y, s["y_bytes"], "y", yt),
        _ptr(pos, s["pos_bytes"], "pos", torch.int32),
        _ptr(topk_w, s["topk_w_bytes"], "topk_w", torch.float32),
        _ptr(partial, s["partial_bytes"], "partial", yt),
        _ptr(slot_rank, s["slot_rank_bytes"], "slot_rank", torch.int32), _stream(stream)))


def combine_reduce_partials(dims: MoeDims, partial, slot_rank, out, stream=None):
    """out[g] = sum of token g's used partial rows."""
    s = buffer_sizes(dims)
    yt = _TORCH_DTYPE[dims.y_dtype]
    _check(lib().moe_combine_reduce_partials(
        ctypes.byref(dims), _ptr(partial, s["partial_bytes"], "partial", yt),
        _ptr(slot_rank, s["slot_rank_bytes"], "slot_rank", torch.int32),
        _ptr(out, s["out_bytes"], "out", yt), _stream(stream)))


def read_status(status, stream=None) -> int:
    """Wait for the stream and return the device status word of dispatch_count."""
    rc = lib().moe_read_status(_ptr(status, 4, "status", torch.int32), _stream(stream))
    if rc == MOE_ERR_CUDA:
        raise MoeError(rc, lib().moe_last_error().decode())
    return rc


def take_device_error(stream=None) -> int:
    """Wait for the stream; return and clear the library's device error word
    (MOE_OK, or MOE_ERR_TIMEOUT if a bounded wait in a kernel gave up)."""
    rc = lib().moe_take_device_error(_stream(stream))
    if rc == MOE_ERR_CUDA:
        raise MoeError(rc, lib().moe_last_error().decode())
    return rc


def selftest_bounded_wait(status, polls: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test: status[0] becomes MOE_OK if
    status[1] turned nonzero within `polls` polls, else MOE_ERR_TIMEOUT."""
    _check(lib().moe_selftest_bounded_wait(_ptr(status, 8, "status", torch.int32), int(polls),
                                           _stream(stream)))


class Buffers:
    """Device buffers for one problem size, allocated with PyTorch.

    ``y`` aliases ``packed_x`` when the expert op keeps the dtype (the
    harness applies it in place); otherwise it is its own allocation.
    """

    def __init__(self, dims: MoeDims, device="cuda", separate_y: bool | None = None):
        self.dims = dims
        s = self.sizes = buffer_sizes(dims)
        N, T, E, R, H = dims.N, dims.T, dims.E, dims.R, dims.H
        NT, cap = N * T, s["cap_rows"]
        i32, f32 = torch.int32, torch.float32
        kw = dict(device=device)
        self.topk_idx = torch.empty(NT, R, dtype=i32, **kw)
        self.topk_w = torch.empty(NT, R, dtype=f32, **kw)
        self.pos = torch.empty(NT, R, dtype=i32, **kw)
        self.expert_counts = torch.empty(E, dtype=i32, **kw)
        self.expert_offsets = torch.empty(E + 1, dtype=i32, **kw)
        self.rank_counts = torch.empty(N, dtype=i32, **kw)
        self.rank_offsets = torch.empty(N + 1, dtype=i32, **kw)
        self.send_counts = torch.empty(N, N, dtype=i32, **kw)
        self.status = torch.zeros(1, dtype=i32, **kw)
        xt = _TORCH_DTYPE[dims.x_dtype]
        self.packed_x = torch.empty(N * cap, H, dtype=xt, **kw)
        spr = H // 128 if dims.x_dtype == MOE_FP8E4M3_BLK128 else 0
        self.packed_scales = torch.empty(N * cap, spr, dtype=f32, **kw) if spr else None
        self.packed_src = torch.empty(N * cap, dtype=i32, **kw)
        if separate_y is None:
            separate_y = dims.x_dtype != dims.y_dtype
        yt = _TORCH_DTYPE[dims.y_dtype]
        self.y = torch.empty(N * cap, H, dtype=yt, **kw) if separate_y else self.packed_x
        self.out = torch.empty(NT, H, dtype=yt, **kw)
