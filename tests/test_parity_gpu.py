"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar: indices, counts, offsets, positions, packed rows and packed_src are
bit-exact; the status word matches; floats meet these tolerances:

* topk_w: relative 2e-6.  The kernel works in f32: the key difference
  z - max z is rounded once (error |z - max| * 2^-24, |z - max| <= 4 for
  selected experts here), expf is within 2 ulp, the softmax denominator is a
  32-lane butterfly over at most 32 sequential terms per lane (<= 32 + 5
  roundings on terms that add up to at most E*ulp-scale but weighted by
  their size -- in practice a few ulp), the division 0.5 ulp, and the
  renormalisation another sum of <= 32 terms (5 levels) and a division.
  Summed, about 20 ulp = 1.2e-6 in the worst realistic case; 2e-6 leaves
  margin while still catching any wrong term.
* combine, bf16 output: |got - ref| <= 2e-2 + 1e-2 |ref| (ref in fp64).
* combine, f32 output: |got - ref| <= 1e-5 * sum_k |w_k y_k|.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_topk_gb300 import workloads as W
from gpu_path import GpuRun, TOPK_W_RTOL, check_combine, compact_of_region
from test_oracle_pins import check_count_invariants

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()
    torch.cuda.init()


def _oracle_route_count(w, inp):
    bias = None if inp.bias is None else inp.bias.numpy()
    idx, tw, _ = oracle.route(inp.logits.numpy(), bias, w.R, w.score_fn, w.renormalize)
    cnt, st = oracle.count(w.N, w.T, w.E, W.default_cap(w), idx)
    return idx, tw, cnt, st


def restore_packed_rows(gr, gpx, gps, gsrc):
    """Put the packed rows the GPU wrote (copied out by packed_rows() and
    already checked) back after the sentinel check, for the expert op and
    combine."""
    b = gr.bufs
    if gr.rows.size == 0:
        return
    dev = b.packed_x.device
    rt = torch.from_numpy(gr.rows).to(dev)
    b.packed_x.view(torch.uint8).view(b.packed_x.shape[0], -1)[rt] = torch.from_numpy(gpx).to(dev)
    b.packed_src[rt] = torch.from_numpy(gsrc).to(dev)
    if gps is not None:
        b.packed_scales[rt] = torch.from_numpy(gps).to(dev)


def _compare(w, inp, topk_idx_override=None, combine_tokens=None, fused=False):
    gr = GpuRun(w, inp, topk_idx_override=topk_idx_override, fused=fused)
    h = gr.host
    idx, tw, cnt, st = _oracle_route_count(w, inp)
    # route (the count input is replaced afterwards when a test overrides it)
    np.testing.assert_allclose(h["topk_w"], tw, rtol=TOPK_W_RTOL, atol=0)
    if topk_idx_override is None:
        np.testing.assert_array_equal(h["topk_idx"], idx)
    else:
        idx = np.ascontiguousarray(topk_idx_override, np.int32)
        np.testing.assert_array_equal(h["topk_idx"], idx)
        cnt, st = oracle.count(w.N, w.T, w.E, W.default_cap(w), idx)
    # count
    assert gr.status == st
    for k in ("expert_counts", "expert_offsets", "rank_counts", "rank_offsets", "send_counts",
              "pos"):
        np.testing.assert_array_equal(h[k], cnt[k], err_msg=k)
    cap = gr.cap
    # pack (only the occupied rows are defined)
    xb = oracle.x_as_bytes(inp.x)
    xs = None if inp.x_scales is None else inp.x_scales.numpy()
    opx, ops, osrc = oracle.pack(xb, xs, cnt["pos"], cnt["rank_offsets"], cap)
    gpx, gps, gsrc = gr.packed_rows()
    crow = compact_of_region(gr.rows, cap, cnt["rank_offsets"])
    np.testing.assert_array_equal(gsrc, osrc[crow])
    np.testing.assert_array_equal(gpx, opx[crow])
    if ops is not None:
        np.testing.assert_array_equal(gps, ops[crow])
    # and nothing else: every other byte of the receive buffers still holds
    # its sentinel (this puts the sentinels back on the occupied rows too)
    gr.assert_untouched_outside_rows()
    # combine (y is recomputed from packed rows, so put them back first)
    restore_packed_rows(gr, gpx, gps, gsrc)
    out = gr.combine()
    y = oracle.expert_op(w.expert_op, opx, ops, osrc, idx, w.H, w.x_dtype, w.y_dtype)
    pos, wt = cnt["pos"], tw
    if combine_tokens is not None:
        pos, wt = pos[combine_tokens], wt[combine_tokens]
    ref, mag = oracle.combine(y, w.y_dtype, pos, cnt["rank_offsets"], wt, cap, w.H)
    check_combine(w, out, ref, mag, combine_tokens)
    return gr, idx, cnt


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_full_size_workload(name):
    """The five workloads at their full sizes, in the launch configuration the
    benchmark uses; every output compared."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    gr, idx, cnt = _compare(w, inp)
    assert gr.status == oracle.OK
    check_count_invariants(w, idx, gr.host, gr.cap)


REDUCED = {
    # ragged everything, f32 rows in and out
    "ragged_f32": W.Workload("ragged_f32", N=3, T=333, E=48, R=6, H=264, x_dtype=W.F32,
                             y_dtype=W.F32, renormalize=True, seed=1),
    # 2 experts per lane (scalar loads), sigmoid + bias, scale expert
    "scalar_lanes": W.Workload("scalar_lanes", N=5, T=77, E=40, R=3, H=136,
                               score_fn=W.SIGMOID, bias="normal",
                               expert_op=W.EXPERT_SCALE, seed=2),
    # largest E and R the library supports
    "max_e_r": W.Workload("max_e_r", N=8, T=40, E=1024, R=32, H=64, renormalize=True, seed=3),
    "r1": W.Workload("r1", N=2, T=100, E=8, R=1, H=128, seed=4),
    "n1": W.Workload("n1", N=1, T=300, E=64, R=4, H=128, seed=5),
    # one expert per rank (E/N < R): the bound uses R
    "e_eq_n": W.Workload("e_eq_n", N=16, T=20, E=16, R=4, H=64, seed=6),
    "t1": W.Workload("t1", N=7, T=1, E=14, R=2, H=64, seed=7),
    "fp8_small": W.Workload("fp8_small", N=4, T=50, E=32, R=4, H=384,
                            x_dtype=W.FP8E4M3_BLK128, expert_op=W.EXPERT_DEQUANT, seed=8),
    # more tokens than one cluster pass: several tiles per block, ragged
    "multi_tile": W.Workload("multi_tile", N=4, T=5000, E=64, R=8, H=64, renormalize=True,
                             seed=9),
    # R > 8 uses the 512-thread count kernel
    "r16": W.Workload("r16", N=4, T=600, E=64, R=16, H=64, score_fn=W.SIGMOID, seed=10),
    # 128 ranks of 2 tokens: a count block's tokens come from so many source
    # ranks that its send counts go to global atomics instead of shared memory
    "many_ranks": W.Workload("many_ranks", N=128, T=2, E=256, R=4, H=64, bias="normal", seed=20),
    # odd E through each count variant (shared-memory tables read as int2 must
    # stay 8-byte aligned): 256-thread blocks, 1024-thread blocks (N*T > 4096)
    # and 512-thread blocks (R > 8)
    "odd_e_256": W.Workload("odd_e_256", N=5, T=100, E=5, R=2, H=64, cap_rows=125, seed=17),
    "odd_e_1024": W.Workload("odd_e_1024", N=3, T=2000, E=21, R=5, H=64, seed=18),
    "odd_e_r17": W.Workload("odd_e_r17", N=1, T=300, E=33, R=17, H=64, score_fn=W.SIGMOID, seed=19),
    # 72 KB bf16 rows: pack and combine run several passes of a 1024-thread
    # block per row, and pack skips its L2 prefetch (rows over 64 KB)
    "wide_rows": W.Workload("wide_rows", N=2, T=24, E=8, R=3, H=36864, renormalize=True,
                            expert_op=W.EXPERT_SCALE, seed=16),
    # bf16 rows, f32 expert outputs
    "bf16_to_f32": W.Workload("bf16_to_f32", N=2, T=64, E=16, R=2, H=512, y_dtype=W.F32,
                              seed=11),
}


@pytest.mark.parametrize("name", list(REDUCED))
def test_reduced_case(name):
    w = REDUCED[name]
    _compare(w, W.make_inputs(w))


def test_ties_break_to_lower_index():
    w = W.WORKLOADS["tiny"].replace(seed=12)
    inp = W.make_inputs(w, tie_every=3)
    _compare(w, inp)


def test_signed_zero_keys_tie():
    w = W.Workload("zeros", N=2, T=32, E=32, R=4, H=64, score_fn=W.SIGMOID, seed=13)
    inp = W.make_inputs(w)
    inp.logits[:, ::2] = -0.0
    inp.logits[:, 1::2] = 0.0
    _compare(w, inp)


def test_capacity_overflow_reports_and_drops():
    w = W.WORKLOADS["tiny"].replace(cap_rows=100, seed=14)
    inp = W.make_inputs(w)
    gr, idx, cnt = _compare(w, inp)
    assert gr.status == oracle.ERR_CAPACITY
    assert (gr.host["pos"] == -1).any()


def test_invalid_expert_ids_are_reported_and_skipped():
    w = W.Workload("bad", N=4, T=64, E=16, R=3, H=64, seed=15)
    inp = W.make_inputs(w)
    bias = None
    idx, _, _ = oracle.route(inp.logits.numpy(), bias, w.R, w.score_fn, w.renormalize)
    bad = idx.copy()
    bad[3, 1] = -1          # below range
    bad[10, 0] = w.E        # above range
    bad[20, 2] = bad[20, 0]  # repeated expert inside one token
    gr, _, cnt = _compare(w, inp, topk_idx_override=bad)
    assert gr.status == oracle.ERR_INVALID
    assert gr.host["pos"][3, 1] == -1 and gr.host["pos"][10, 0] == -1
    assert gr.host["pos"][20, 2] == -1 and gr.host["pos"][20, 0] >= 0


def test_empty_batch():
    import combine_moe_route_topk_gb300 as moe
    w = W.Workload("empty", N=4, T=0, E=16, R=2, H=64)
    dims = moe.dims_of(w)
    b = moe.Buffers(dims)
    b.expert_counts.fill_(7)
    b.send_counts.fill_(7)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    logits = torch.empty(0, 16, dtype=torch.float32, device="cuda")
    moe.route_topk(dims, logits, None, W.SOFTMAX, False, b.topk_idx, b.topk_w)
    moe.dispatch_count(dims, b.topk_idx, b.expert_counts, b.expert_offsets, b.rank_counts,
                       b.rank_offsets, b.send_counts, b.pos, b.status)
    moe.dispatch_pack(dims, x, None, b.pos, b.packed_x, None, b.packed_src)
    moe.combine(dims, b.y, b.pos, b.topk_w, b.out)
    assert moe.read_status(b.status) == moe.MOE_OK
    assert int(b.expert_counts.abs().sum()) == 0 and int(b.send_counts.abs().sum()) == 0
    assert b.expert_offsets.cpu().tolist() == [0] * 17
    assert b.rank_offsets.cpu().tolist() == [0] * 5


def test_repeated_calls_are_deterministic():
    """Same inputs twice -> identical bytes (no scheduling dependence)."""
    w = W.WORKLOADS["kimi_k2_decode"].replace(H=256)
    inp = W.make_inputs(w)
    a = GpuRun(w, inp)
    b = GpuRun(w, inp)
    for k in a.host:
        np.testing.assert_array_equal(a.host[k], b.host[k], err_msg=k)
    pa, _, sa = a.packed_rows()
    pb, _, sb = b.packed_rows()
    np.testing.assert_array_equal(pa, pb)
    np.testing.assert_array_equal(sa, sb)
    oa, ob = a.combine().cpu(), b.combine().cpu()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))


def test_cuda_graph_capture_and_replay():
    """The four calls capture into one CUDA graph (fixed grids, no host
    synchronisation) and the replay recomputes everything for new inputs."""
    import combine_moe_route_topk_gb300 as moe
    w = W.WORKLOADS["tiny"]
    dims = moe.dims_of(w)
    b = moe.Buffers(dims)
    inp = W.make_inputs(w, device="cuda")
    logits, x = inp.logits.clone(), inp.x.clone()

    def calls():
        moe.route_topk(dims, logits, None, w.score_fn, w.renormalize, b.topk_idx, b.topk_w)
        moe.dispatch_count(dims, b.topk_idx, b.expert_counts, b.expert_offsets, b.rank_counts,
                           b.rank_offsets, b.send_counts, b.pos, b.status)
        moe.dispatch_pack(dims, x, None, b.pos, b.packed_x, None, b.packed_src)
        moe.combine(dims, b.y, b.pos, b.topk_w, b.out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()
    w2 = w.replace(seed=99)
    inp2 = W.make_inputs(w2)
    logits.copy_(inp2.logits)
    x.copy_(inp2.x)
    b.out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert moe.read_status(b.status) == moe.MOE_OK
    ref = oracle.run(w2, inp2)
    np.testing.assert_array_equal(b.topk_idx.cpu().numpy(), ref["topk_idx"])
    np.testing.assert_array_equal(b.pos.cpu().numpy(), ref["pos"])
    check_combine(w2, b.out, ref["out"], ref["mag"])


def test_device_error_word_is_clear_after_normal_runs():
    import combine_moe_route_topk_gb300 as moe
    w = W.WORKLOADS["tiny"]
    GpuRun(w, W.make_inputs(w)).combine()
    assert moe.take_device_error() == moe.MOE_OK


def test_bulk_pack_kernel_matches_too():
    """The bulk-copy pack kernel (MOE_PACK_KERNEL=bulk) gives the same bytes;
    run in a child process because the choice is read once."""
    import os
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, 'tests'); sys.path.insert(0, '.');"
        "import numpy as np, oracle;"
        "from combine_moe_route_topk_gb300 import workloads as W;"
        "from gpu_path import GpuRun, compact_of_region;"
        "ok = True\n"
        "for name in ('tiny', 'skewed'):\n"
        "    w = W.WORKLOADS[name]; inp = W.make_inputs(w); gr = GpuRun(w, inp)\n"
        "    ref = oracle.run(w, inp, with_combine=False)\n"
        "    px, ps, src = gr.packed_rows(); c = compact_of_region(gr.rows, gr.cap, ref['rank_offsets'])\n"
        "    ok &= np.array_equal(px, ref['packed_x'][c]) and np.array_equal(src, ref['packed_src'][c])\n"
        "    ok &= ps is None or np.array_equal(ps, ref['packed_scales'][c])\n"
        "import combine_moe_route_topk_gb300 as moe\n"
        "ok &= moe.take_device_error() == moe.MOE_OK\n"
        "print('BULK_OK' if ok else 'BULK_MISMATCH')\n")
    env = dict(os.environ, MOE_PACK_KERNEL="bulk")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                       text=True, timeout=600)
    assert "BULK_OK" in r.stdout, r.stdout + r.stderr
