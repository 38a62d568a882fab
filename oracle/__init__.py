"""CPU oracle for MoE token routing (test infrastructure only).

Thin ctypes wrapper over ``moe_oracle.c``: a plain single-threaded C
statement of route top-k, dispatch count, dispatch pack, the harness expert
op and combine.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use this package; the GPU library never does,
and this package never imports the GPU library.

Every function takes and returns numpy arrays.  Pack, expert op and combine
work on *compact* rows: the receive-region row ``pos = d*cap + local`` is
stored at compact row ``rank_offsets[d] + local``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_INVALID, ERR_CAPACITY = 0, -1, -4
SOFTMAX, SIGMOID = 0, 1
BIAS_SELECT_ONLY = 0x10  # flag OR'ed into score_fn: bias in the selection key only
BF16, F32, FP8 = 0, 1, 2
EXPERT_OPS = {"identity": 0, "scale": 1, "dequant": 2}


def build_lib(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (plain -O2, IEEE arithmetic)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_lib()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int
            lib.oracle_route.argtypes = [i64, i32, i32, P, P, i32, i32, P, P, P]
            lib.oracle_count.argtypes = [i32, i64, i32, i32, i64, P, P, P, P, P, P, P]
            lib.oracle_pack.argtypes = [i64, i32, i64, i64, i64, P, P, P, P, P, P, P]
            lib.oracle_expert_op.argtypes = [i32, i64, i64, i32, i32, P, P, P, P, P]
            lib.oracle_combine.argtypes = [i64, i32, i64, i32, i64, P, P, P, P, P, P]
            lib.oracle_fp8e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_fp8e4m3_decode.restype = ctypes.c_double
            lib.oracle_f32_to_fp8e4m3.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_fp8e4m3.restype = ctypes.c_uint8
            lib.oracle_quantize_rows.argtypes = [i64, i64, P, P, P]
            lib.oracle_combine_rank.argtypes = [i64, i32, i64, i32, i64, i32, P, P, P, P, P]
            lib.oracle_combine_partials.argtypes = [i64, i32, i32, i64, i32, i64, P, P, P, P, P, P]
            lib.oracle_reduce_partials.argtypes = [i64, i32, i64, i32, P, P, P]
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def route(logits, bias, R, score_fn, renorm):
    """Top-R experts and weights per token. Returns (idx i32, w f32, w f64)."""
    lib = _load()
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    NT, E = logits.shape
    idx = np.empty((NT, R), np.int32)
    w = np.empty((NT, R), np.float32)
    w64 = np.empty((NT, R), np.float64)
    rc = lib.oracle_route(NT, E, R, _p(logits), _p(bias), int(score_fn), int(bool(renorm)),
                          _p(idx), _p(w), _p(w64))
    if rc != OK:
        raise ValueError(f"oracle_route rejected its arguments ({rc})")
    return idx, w, w64


def count(N, T, E, cap, topk_idx):
    """Counts, offsets and positions. Returns (dict of arrays, status)."""
    lib = _load()
    topk_idx = _c(topk_idx, np.int32)
    R = topk_idx.shape[1]
    out = {
        "expert_counts": np.empty(E, np.int32),
        "expert_offsets": np.empty(E + 1, np.int32),
        "rank_counts": np.empty(N, np.int32),
        "rank_offsets": np.empty(N + 1, np.int32),
        "send_counts": np.empty((N, N), np.int32),
        "pos": np.empty((N * T, R), np.int32),
    }
    st = lib.oracle_count(N, T, E, R, cap, _p(topk_idx), _p(out["expert_counts"]),
                          _p(out["expert_offsets"]), _p(out["rank_counts"]),
                          _p(out["rank_offsets"]), _p(out["send_counts"]), _p(out["pos"]))
    return out, st


def pack(x_bytes, x_scales, pos, rank_offsets, cap):
    """Compact packed rows. ``x_bytes`` is uint8 [NT, row_bytes]."""
    lib = _load()
    x_bytes = _c(x_bytes, np.uint8)
    x_scales = _c(x_scales, np.float32)
    pos = _c(pos, np.int32)
    rank_offsets = _c(rank_offsets, np.int32)
    NT, rb = x_bytes.shape
    R = pos.shape[1]
    rows = int(rank_offsets[-1])
    spr = 0 if x_scales is None else x_scales.shape[1]
    packed_x = np.zeros((rows, rb), np.uint8)
    packed_scales = np.zeros((rows, spr), np.float32) if spr else None
    packed_src = np.full(rows, -1, np.int32)
    lib.oracle_pack(NT, R, rb, spr, cap, _p(x_bytes), _p(x_scales), _p(pos),
                    _p(rank_offsets), _p(packed_x), _p(packed_scales), _p(packed_src))
    return packed_x, packed_scales, packed_src


def expert_op(op, packed_x, packed_scales, packed_src, topk_idx, H, x_dtype, y_dtype):
    """Harness expert op on compact rows; returns y as uint16 (bf16) or f32."""
    lib = _load()
    rows = packed_src.shape[0]
    y = np.zeros((rows, H), np.uint16 if y_dtype == BF16 else np.float32)
    packed_x = _c(packed_x, np.uint8)
    lib.oracle_expert_op(EXPERT_OPS[op], rows, H, x_dtype, y_dtype, _p(packed_x),
                         _p(_c(packed_scales, np.float32)), _p(_c(packed_src, np.int32)),
                         _p(_c(topk_idx, np.int32)), _p(y))
    return y


def combine(y, y_dtype, pos, rank_offsets, topk_w, cap, H):
    """out[g] = sum_k w[g][k] * y[pos[g][k]] in double; also sum_k |w*y|."""
    lib = _load()
    pos = _c(pos, np.int32)
    NT, R = pos.shape
    out = np.empty((NT, H), np.float64)
    mag = np.empty((NT, H), np.float64)
    y = np.ascontiguousarray(y)
    lib.oracle_combine(NT, R, H, y_dtype, cap, _p(y), _p(pos), _p(_c(rank_offsets, np.int32)),
                       _p(_c(topk_w, np.float32)), _p(out), _p(mag))
    return out, mag


def combine_rank(y, y_dtype, pos, rank_offsets, topk_w, cap, H, rank):
    """Local accumulation of one rank: sum of w*y over the token's pairs on
    `rank` (0 where there are none), in double."""
    lib = _load()
    pos = _c(pos, np.int32)
    NT, R = pos.shape
    out = np.empty((NT, H), np.float64)
    lib.oracle_combine_rank(NT, R, H, y_dtype, cap, rank, _p(np.ascontiguousarray(y)), _p(pos),
                            _p(_c(rank_offsets, np.int32)), _p(_c(topk_w, np.float32)), _p(out))
    return out


def combine_partials(y, y_dtype, pos, rank_offsets, topk_w, cap, H, N):
    """Per (token, distinct destination rank) partial rows rounded to y_dtype.
    Returns (partial [NT, P, H], slot_rank i32 [NT, P]) with P = min(R, N)."""
    lib = _load()
    pos = _c(pos, np.int32)
    NT, R = pos.shape
    P = min(R, N)
    partial = np.zeros((NT, P, H), np.uint16 if y_dtype == BF16 else np.float32)
    slot_rank = np.empty((NT, P), np.int32)
    lib.oracle_combine_partials(NT, R, P, H, y_dtype, cap, _p(np.ascontiguousarray(y)), _p(pos),
                                _p(_c(rank_offsets, np.int32)), _p(_c(topk_w, np.float32)),
                                _p(partial), _p(slot_rank))
    return partial, slot_rank


def reduce_partials(partial, slot_rank, y_dtype):
    """out[g] = sum of the used partial rows of token g, in double."""
    lib = _load()
    NT, P, H = partial.shape
    out = np.empty((NT, H), np.float64)
    lib.oracle_reduce_partials(NT, P, H, y_dtype, _p(np.ascontiguousarray(partial)),
                               _p(_c(slot_rank, np.int32)), _p(out))
    return out


def fp8e4m3_decode(code: int) -> float:
    return _load().oracle_fp8e4m3_decode(code)


def f32_to_fp8e4m3(v: float) -> int:
    return _load().oracle_f32_to_fp8e4m3(v)


def quantize_rows(x_bf16_rows):
    """Block fp8 quantisation of bf16 rows (uint16 bits or a bf16 tensor):
    returns (codes uint8 [rows, H], scales f32 [rows, H/128])."""
    lib = _load()
    if hasattr(x_bf16_rows, "numpy"):
        import torch
        x_bf16_rows = x_bf16_rows.contiguous().view(torch.int16).numpy().view(np.uint16)
    x = np.ascontiguousarray(x_bf16_rows, dtype=np.uint16)
    rows, H = x.shape
    codes = np.empty((rows, H), np.uint8)
    scales = np.empty((rows, H // 128), np.float32)
    rc = lib.oracle_quantize_rows(rows, H, _p(x), _p(codes), _p(scales))
    if rc != OK:
        raise ValueError("H must be a multiple of 128")
    return codes, scales


def f32_to_bf16_bits(v: float) -> int:
    return _load().oracle_f32_to_bf16(v)


def x_as_bytes(x):
    """View a CPU torch tensor or numpy array of rows as uint8 [rows, bytes]."""
    if hasattr(x, "numpy"):
        import torch
        t = x.contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        a = t.numpy()
    else:
        a = np.ascontiguousarray(x)
    # the row width is explicit so that an empty batch keeps its shape (0, bytes)
    return a.view(np.uint8).reshape(a.shape[0], a.dtype.itemsize * int(np.prod(a.shape[1:])))


def run(w, inp, with_combine=True):
    """Whole path for one workload (``combine_moe_route_topk_gb300.workloads``)."""
    logits = inp.logits.numpy()
    bias = None if inp.bias is None else inp.bias.numpy()
    idx, tw, tw64 = route(logits, bias, w.R, w.score_fn, w.renormalize)
    cap = w.cap_rows if w.cap_rows > 0 else w.N * w.T * max(w.R, w.E // w.N)
    cnt, st = count(w.N, w.T, w.E, cap, idx)
    xs = None if inp.x_scales is None else inp.x_scales.numpy()
    px, ps, psrc = pack(x_as_bytes(inp.x), xs, cnt["pos"], cnt["rank_offsets"], cap)
    res = dict(topk_idx=idx, topk_w=tw, topk_w64=tw64, status=st, cap=cap,
               packed_x=px, packed_scales=ps, packed_src=psrc, **cnt)
    if with_combine:
        y = expert_op(w.expert_op, px, ps, psrc, idx, w.H, w.x_dtype, w.y_dtype)
        out, mag = combine(y, w.y_dtype, cnt["pos"], cnt["rank_offsets"], tw, cap, w.H)
        res.update(y=y, out=out, mag=mag)
    return res
