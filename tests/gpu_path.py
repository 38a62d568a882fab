"""Test harness: run the CUDA path through the C ABI and compare with the oracle.

The expert op between pack and combine (identity / per-expert scale / fp8
dequant) stands in for the grouped expert GEMM and is applied here with
plain PyTorch on the GPU; it is not part of the library.
"""
from __future__ import annotations

import numpy as np
import torch

import combine_moe_route_topk_gb300 as moe
import oracle
from combine_moe_route_topk_gb300 import workloads as W

# Tolerances (see the test modules for their derivation)
TOPK_W_RTOL = 2e-6
BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_RTOL_OF_MAG = 1e-5


def occupied_rows(rank_counts: np.ndarray, cap: int) -> np.ndarray:
    """Receive-region rows that dispatch wrote, in region order."""
    parts = [np.arange(d * cap, d * cap + min(int(c), cap)) for d, c in enumerate(rank_counts)]
    return np.concatenate(parts) if parts else np.zeros(0, np.int64)


def compact_of_region(rows: np.ndarray, cap: int, rank_offsets: np.ndarray) -> np.ndarray:
    return rank_offsets[rows // cap] + rows % cap


def expert_op_gpu(w: W.Workload, bufs: moe.Buffers, rows: torch.Tensor) -> None:
    """Apply the harness expert op to the occupied rows, writing bufs.y."""
    if rows.numel() == 0:
        return
    if w.expert_op == W.EXPERT_IDENTITY:
        if bufs.y.data_ptr() != bufs.packed_x.data_ptr():
            bufs.y[rows] = bufs.packed_x[rows].to(bufs.y.dtype)
        return
    if w.expert_op == W.EXPERT_SCALE:
        src = bufs.packed_src[rows].long()
        e = bufs.topk_idx.view(-1)[src].long()
        s = (1.0 + ((e % 7) - 3).to(torch.float32) / 16.0).unsqueeze(1)
        bufs.y[rows] = (bufs.packed_x[rows].to(torch.float32) * s).to(bufs.y.dtype)
        return
    if w.expert_op == W.EXPERT_DEQUANT:
        q = bufs.packed_x[rows].view(torch.float8_e4m3fn).to(torch.float32)
        sc = bufs.packed_scales[rows].repeat_interleave(128, dim=1)
        bufs.y[rows] = (q * sc).to(bufs.y.dtype)
        return
    raise ValueError(w.expert_op)


SENTINEL_BYTE = 0xA5  # packed_x / packed_scales bytes before a pack
SENTINEL_SRC = -7     # packed_src entries before a pack


def fill_sentinels(packed_x: torch.Tensor, packed_scales: torch.Tensor | None,
                   packed_src: torch.Tensor, rows: torch.Tensor | None = None) -> None:
    """Set the receive buffers (or only `rows` of them) to the sentinels."""
    for t in (packed_x, packed_scales):
        if t is not None:
            if rows is None:
                t.view(torch.uint8).fill_(SENTINEL_BYTE)
            elif rows.numel():
                t.view(torch.uint8).view(t.shape[0], -1)[rows] = SENTINEL_BYTE
    if rows is None:
        packed_src.fill_(SENTINEL_SRC)
    elif rows.numel():
        packed_src[rows] = SENTINEL_SRC


def _all_bytes_equal(t: torch.Tensor, byte: int) -> bool:
    """Every byte of t equals `byte` (checked on the device, 1 GB at a time)."""
    flat = t.reshape(-1).view(torch.uint8)
    step = 1 << 30
    for i in range(0, flat.numel(), step):
        if not bool((flat[i:i + step] == byte).all()):
            return False
    return True


def assert_untouched_outside(rows: np.ndarray, packed_x: torch.Tensor,
                             packed_scales: torch.Tensor | None, packed_src: torch.Tensor) -> None:
    """After the occupied `rows` have been checked: put the sentinels back on
    them and require every byte of the receive buffers to be a sentinel, i.e.
    dispatch wrote nothing outside the rows it owns (no stray store into the
    unused tail of a rank region or past it)."""
    rt = torch.from_numpy(np.ascontiguousarray(rows, np.int64)).to(packed_x.device)
    fill_sentinels(packed_x, packed_scales, packed_src, rt)
    assert _all_bytes_equal(packed_x, SENTINEL_BYTE), "packed_x written outside the occupied rows"
    if packed_scales is not None:
        assert _all_bytes_equal(packed_scales, SENTINEL_BYTE), \
            "packed_scales written outside the occupied rows"
    assert bool((packed_src == SENTINEL_SRC).all()), "packed_src written outside the occupied rows"


class GpuRun:
    """Route -> count -> pack -> (expert op) -> combine on the current GPU.

    The receive buffers start filled with sentinels, so that a test can check
    that dispatch wrote nothing outside the occupied rows."""

    def __init__(self, w: W.Workload, inp: W.Inputs, topk_idx_override: np.ndarray | None = None,
                 fused: bool = False):
        self.w = w
        self.dims = moe.dims_of(w)
        dev = torch.device("cuda", torch.cuda.current_device())
        self.d = W.Inputs(*(t.to(dev) if t is not None else None
                            for t in (inp.logits, inp.bias, inp.x, inp.x_scales)))
        self.bufs = moe.Buffers(self.dims, device=dev)
        b = self.bufs
        fill_sentinels(b.packed_x, b.packed_scales, b.packed_src)
        if fused:
            assert topk_idx_override is None
            ws = torch.zeros(b.sizes["fused_workspace_bytes"], dtype=torch.uint8, device=dev)
            moe.dispatch_fused(self.dims, self.d.logits, self.d.bias, w.score_fn, w.renormalize,
                               self.d.x, self.d.x_scales, b.topk_idx, b.topk_w, b.expert_counts,
                               b.expert_offsets, b.rank_counts, b.rank_offsets, b.send_counts,
                               b.pos, b.status, b.packed_x, b.packed_scales, b.packed_src, ws)
        else:
            moe.route_topk(self.dims, self.d.logits, self.d.bias, w.score_fn, w.renormalize,
                           b.topk_idx, b.topk_w)
            if topk_idx_override is not None:
                b.topk_idx.copy_(torch.from_numpy(np.ascontiguousarray(topk_idx_override)))
            moe.dispatch_count(self.dims, b.topk_idx, b.expert_counts, b.expert_offsets,
                               b.rank_counts, b.rank_offsets, b.send_counts, b.pos, b.status)
            moe.dispatch_pack(self.dims, self.d.x, self.d.x_scales, b.pos, b.packed_x,
                              b.packed_scales, b.packed_src)
        self.status = moe.read_status(b.status)
        self.cap = b.sizes["cap_rows"]
        self.host = {k: getattr(b, k).cpu().numpy() for k in
                     ("topk_idx", "topk_w", "pos", "expert_counts", "expert_offsets",
                      "rank_counts", "rank_offsets", "send_counts")}
        self.rows = occupied_rows(self.host["rank_counts"], self.cap)

    def assert_untouched_outside_rows(self):
        """Nothing but the occupied rows of the receive buffers was written.
        Resets those rows to the sentinels: call after packed_rows(), before
        combine()."""
        b = self.bufs
        assert_untouched_outside(self.rows, b.packed_x, b.packed_scales, b.packed_src)

    def packed_rows(self):
        rows = torch.from_numpy(self.rows).to(self.bufs.packed_x.device)
        px = oracle.x_as_bytes(self.bufs.packed_x[rows].cpu())
        ps = None if self.bufs.packed_scales is None else self.bufs.packed_scales[rows].cpu().numpy()
        src = self.bufs.packed_src[rows].cpu().numpy()
        return px, ps, src

    def combine(self) -> torch.Tensor:
        rows = torch.from_numpy(self.rows).to(self.bufs.packed_x.device)
        expert_op_gpu(self.w, self.bufs, rows)
        moe.combine(self.dims, self.bufs.y, self.bufs.pos, self.bufs.topk_w, self.bufs.out)
        torch.cuda.synchronize()
        return self.bufs.out


def check_combine(w: W.Workload, got: torch.Tensor, ref: np.ndarray, mag: np.ndarray,
                  tokens: np.ndarray | None = None) -> None:
    g = got.cpu()
    if tokens is not None:
        g = g[torch.from_numpy(tokens)]
    g = g.to(torch.float64).numpy()
    err = np.abs(g - ref)
    if w.y_dtype == W.BF16:
        lim = BF16_ATOL + BF16_RTOL * np.abs(ref)
    else:
        lim = F32_RTOL_OF_MAG * mag + 1e-30
    bad = ~(err <= lim)  # NaN (e.g. an unwritten sentinel) fails too
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"combine mismatch at {tuple(i)}: got {g[tuple(i)]!r} ref {ref[tuple(i)]!r} "
                             f"({int(bad.sum())} elements out of tolerance)")
