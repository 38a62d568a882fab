"""Parity of the rank-restricted pack, the per-rank local accumulation and
the send-side partial accumulation (partials + reduction) with the oracle.

Tolerances are the combine's: bf16 outputs |got - ref| <= 2e-2 + 1e-2|ref|,
f32 outputs <= 1e-5 * sum|w y|.  A bf16 partial row is one rounding of an
f32 sum on the GPU and of the double sum (via float) in the oracle, so it
may differ by one bf16 step, well inside the bf16 tolerance; slot ranks and
packed rows are compared exactly.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_topk_gb300 as moe
import oracle
from combine_moe_route_topk_gb300 import workloads as W
from gpu_path import GpuRun, check_combine, compact_of_region, expert_op_gpu, occupied_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()


CASES = {
    "dsv3": W.WORKLOADS["dsv3_decode"],
    "qwen_small": W.WORKLOADS["qwen3_235b_prefill"].replace(T=512, H=1024),
    "tiny": W.WORKLOADS["tiny"],
    "r16_f32": W.Workload("r16_f32", N=4, T=100, E=64, R=16, H=64, x_dtype=W.F32,
                          y_dtype=W.F32, expert_op=W.EXPERT_SCALE, seed=51),
    # row widths that are not powers of two (66 and 25 vectors) and a
    # token count that is not a multiple of the 8 tokens of a rank-local block
    "odd_f32": W.Workload("odd_f32", N=3, T=333, E=48, R=6, H=264, x_dtype=W.F32,
                          y_dtype=W.F32, seed=52),
    "odd_bf16": W.Workload("odd_bf16", N=5, T=77, E=40, R=3, H=200, seed=53),
    # fp8 rows with block scales through the rank-restricted pack
    "fp8": W.Workload("fp8", N=4, T=50, E=32, R=4, H=384, x_dtype=W.FP8E4M3_BLK128,
                      expert_op=W.EXPERT_DEQUANT, seed=54),
}


def _setup(w):
    inp = W.make_inputs(w)
    gr = GpuRun(w, inp)
    ref = oracle.run(w, inp)
    assert gr.status == oracle.OK
    dev = gr.bufs.packed_x.device
    rows = torch.from_numpy(gr.rows).to(dev)
    expert_op_gpu(w, gr.bufs, rows)  # y for every occupied row
    torch.cuda.synchronize()
    return inp, gr, ref


@pytest.mark.parametrize("name", ["tiny", "qwen_small", "odd_f32", "odd_bf16", "fp8"])
def test_pack_rank_writes_only_that_region(name):
    check_pack_rank(CASES[name])


def check_pack_rank(w):
    """Each rank's rows equal the oracle's, and nothing outside them is written
    (every rank for N <= 8, else the first, second, middle and last)."""
    inp = W.make_inputs(w)
    gr = GpuRun(w, inp)
    ref = oracle.run(w, inp, with_combine=False)
    b, cap = gr.bufs, gr.cap
    ranks = range(w.N) if w.N <= 8 else [0, 1, w.N // 2, w.N - 1]
    for d in ranks:
        b.packed_x.view(torch.uint8).fill_(0xA5)
        b.packed_src.fill_(-7)
        moe.dispatch_pack_rank(gr.dims, d, gr.d.x, gr.d.x_scales, b.pos, b.packed_x,
                               b.packed_scales, b.packed_src)
        torch.cuda.synchronize()
        n_d = int(ref["rank_counts"][d])
        rows = np.arange(d * cap, d * cap + min(n_d, cap))
        crow = compact_of_region(rows, cap, ref["rank_offsets"])
        rt = torch.from_numpy(rows).to(b.packed_x.device)
        np.testing.assert_array_equal(oracle.x_as_bytes(b.packed_x[rt].cpu()), ref["packed_x"][crow],
                                      err_msg=f"rank {d}")
        np.testing.assert_array_equal(b.packed_src[rt].cpu().numpy(), ref["packed_src"][crow],
                                      err_msg=f"rank {d}")
        if b.packed_scales is not None:
            np.testing.assert_array_equal(b.packed_scales[rt].cpu().numpy(),
                                          ref["packed_scales"][crow], err_msg=f"rank {d}")
        others = torch.ones(b.packed_src.numel(), dtype=torch.bool, device=rt.device)
        others[rt] = False
        assert bool((b.packed_src[others] == -7).all()), f"rank {d}"


@pytest.mark.parametrize("name", list(CASES))
def test_local_accumulation_per_rank(name):
    check_local_accumulation(CASES[name])


def rank_magnitude(w, ref, d):
    """sum |w * y| over the pairs of each token that land on rank d: the
    magnitude that bounds the rounding error of rank d's local sum (f32
    tolerance 1e-5 of it).  The whole combine's magnitude would be up to R
    times larger for a token with one pair on d, and the tolerance as loose."""
    pos_d = np.where(ref["pos"] // ref["cap"] == d, ref["pos"], -1).astype(np.int32)
    _, mag_d = oracle.combine(ref["y"], w.y_dtype, pos_d, ref["rank_offsets"], ref["topk_w"],
                              ref["cap"], w.H)
    return mag_d


def check_local_accumulation(w):
    """Each rank's local sum against the oracle; all ranks add up to the combine."""
    inp, gr, ref = _setup(w)
    b = gr.bufs
    out_d = torch.empty_like(b.out)
    total = torch.zeros(b.out.shape, dtype=torch.float64, device=b.out.device)
    ranks = range(w.N) if w.N <= 8 else [0, 1, w.N // 2, w.N - 1]
    for d in ranks:
        out_d.view(torch.uint8).fill_(0xFF)  # NaN: every output row must be written
        moe.combine_rank(gr.dims, d, b.y, b.pos, b.topk_w, out_d)
        torch.cuda.synchronize()
        want = oracle.combine_rank(ref["y"], w.y_dtype, ref["pos"], ref["rank_offsets"],
                                   ref["topk_w"], ref["cap"], w.H, d)
        check_combine(w, out_d, want, rank_magnitude(w, ref, d))
        total += out_d.to(torch.float64)
    if len(ranks) == w.N:
        # the all-reduce over ranks (not part of the library) gives the combine
        tot = total.cpu().numpy()
        lim = (w.N * (2e-2 + 1e-2 * np.abs(ref["out"])) if w.y_dtype == W.BF16
               else 1e-5 * ref["mag"] * w.N + 1e-30)
        assert (np.abs(tot - ref["out"]) <= lim).all()


@pytest.mark.parametrize("name", list(CASES))
def test_send_side_partials_and_reduction(name):
    check_send_side_partials(CASES[name])


def check_send_side_partials(w):
    """Partial rows and slots against the oracle; their reduction against the
    oracle's and against the plain combine."""
    inp, gr, ref = _setup(w)
    b = gr.bufs
    s = moe.buffer_sizes(gr.dims)
    P = s["partial_slots"]
    yt = b.y.dtype
    partial = torch.empty(w.NT, P, w.H, dtype=yt, device=b.y.device)
    slot_rank = torch.empty(w.NT, P, dtype=torch.int32, device=b.y.device)
    moe.combine_partials(gr.dims, b.y, b.pos, b.topk_w, partial, slot_rank)
    out = torch.empty_like(b.out)
    moe.combine_reduce_partials(gr.dims, partial, slot_rank, out)
    torch.cuda.synchronize()
    opart, oslot = oracle.combine_partials(ref["y"], w.y_dtype, ref["pos"], ref["rank_offsets"],
                                           ref["topk_w"], ref["cap"], w.H, w.N)
    np.testing.assert_array_equal(slot_rank.cpu().numpy(), oslot)
    gp = partial.cpu().to(torch.float64).numpy()
    if w.y_dtype == W.BF16:
        op = torch.from_numpy(opart.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        assert (np.abs(gp - op) <= 2e-2 + 1e-2 * np.abs(op)).all()
    else:
        np.testing.assert_allclose(gp, opart, rtol=1e-5, atol=1e-6)
    # reduction of the oracle's partials, and closeness to the plain combine
    oref = oracle.reduce_partials(opart, oslot, w.y_dtype)
    check_combine(w, out, oref, ref["mag"])
    check_combine(w, out, ref["out"], ref["mag"] * 2)
