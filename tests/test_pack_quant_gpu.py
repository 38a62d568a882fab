"""Parity of the quantising pack (bf16 rows -> e4m3 codes + per-128 scales)
with the oracle: codes, scales and packed_src bit-exact on the occupied rows,
and every other byte of the three buffers left as it was (sentinels).

Both sides take every rounding decision in the same precision: amax is exact,
scale = fl32(amax / 448), the quotient fl32(x / scale) is IEEE-rounded on
both sides, and the e4m3 rounding (nearest, ties to even, saturating) is the
format's; the oracle's encoder is pinned in test_oracle_pins.py.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_topk_gb300 as moe
import oracle
from combine_moe_route_topk_gb300 import workloads as W
from gpu_path import assert_untouched_outside, compact_of_region, fill_sentinels, occupied_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()


def _run(w, inp, special=None, fused=False):
    """fused: moe_dispatch_fused_quant (route, count and the quantising pack
    in one call) in place of the three calls; its routing, counts and rows are
    checked against the oracle as well."""
    dims = moe.dims_of(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    b = moe.Buffers(dims, device=dev)
    logits = inp.logits.to(dev)
    bias = None if inp.bias is None else inp.bias.to(dev)
    x = inp.x.to(dev)
    q = moe.buffer_sizes(moe.fp8_dims(dims))
    packed_q = torch.empty(q["packed_x_bytes"], dtype=torch.uint8, device=dev)
    packed_scales = torch.empty(q["packed_scales_bytes"] // 4, dtype=torch.float32, device=dev)
    pq2 = packed_q.view(-1, w.H)
    ps2 = packed_scales.view(-1, w.H // 128)
    fill_sentinels(pq2, ps2, b.packed_src)
    if fused:
        ws = torch.zeros(b.sizes["fused_workspace_bytes"], dtype=torch.uint8, device=dev)
        moe.dispatch_fused_quant(dims, logits, bias, w.score_fn, w.renormalize, x, b.topk_idx,
                                 b.topk_w, b.expert_counts, b.expert_offsets, b.rank_counts,
                                 b.rank_offsets, b.send_counts, b.pos, b.status, packed_q,
                                 packed_scales, b.packed_src, ws)
    else:
        moe.route_topk(dims, logits, bias, w.score_fn, w.renormalize, b.topk_idx, b.topk_w)
        moe.dispatch_count(dims, b.topk_idx, b.expert_counts, b.expert_offsets, b.rank_counts,
                           b.rank_offsets, b.send_counts, b.pos, b.status)
        moe.dispatch_pack_quant(dims, x, b.pos, packed_q, packed_scales, b.packed_src)
    assert moe.read_status(b.status) == moe.MOE_OK
    cap = b.sizes["cap_rows"]
    rank_counts = b.rank_counts.cpu().numpy()
    rows = occupied_rows(rank_counts, cap)
    rows_t = torch.from_numpy(rows).to(dev)
    gq = packed_q.view(-1, w.H)[rows_t].cpu().numpy()
    gs = packed_scales.view(-1, w.H // 128)[rows_t].cpu().numpy()
    gsrc = b.packed_src[rows_t].cpu().numpy()
    # oracle: quantise every token row, then pack the fp8 rows
    idx, _, _ = oracle.route(inp.logits.numpy(), None if inp.bias is None else inp.bias.numpy(),
                             w.R, w.score_fn, w.renormalize)
    cnt, st = oracle.count(w.N, w.T, w.E, cap, idx)
    assert st == oracle.OK
    if fused:
        np.testing.assert_array_equal(b.topk_idx.cpu().numpy(), idx)
        for k in ("expert_counts", "expert_offsets", "rank_counts", "rank_offsets", "send_counts", "pos"):
            np.testing.assert_array_equal(getattr(b, k).cpu().numpy(), cnt[k], err_msg=k)
    codes, scales = oracle.quantize_rows(inp.x)
    oq, osc, osrc = oracle.pack(codes, scales, cnt["pos"], cnt["rank_offsets"], cap)
    crow = compact_of_region(rows, cap, cnt["rank_offsets"])
    np.testing.assert_array_equal(gsrc, osrc[crow])
    np.testing.assert_array_equal(gs.view(np.uint32), osc[crow].view(np.uint32))
    bad = np.argwhere(gq != oq[crow])
    assert bad.size == 0, (f"{len(bad)} codes differ, first at {tuple(bad[0])}: "
                           f"got {gq[tuple(bad[0])]:#04x} want {oq[crow][tuple(bad[0])]:#04x}")
    # nothing outside the occupied rows was written
    assert_untouched_outside(rows, pq2, ps2, b.packed_src)


def test_quant_pack_full_size_dsv3():
    w = W.WORKLOADS["dsv3_decode"]
    _run(w, W.make_inputs(w))


def test_quant_pack_full_size_kimi():
    w = W.WORKLOADS["kimi_k2_decode"]
    _run(w, W.make_inputs(w))


# the last shape has 72 KB rows: 2304 chunks per row, more than one pass of a
# 1024-thread block, and too wide for the L2 prefetch of x
@pytest.mark.parametrize("N,T,E,R,H", [(3, 77, 24, 3, 128), (4, 50, 32, 5, 384),
                                       (2, 300, 16, 2, 1152), (2, 24, 8, 3, 36864)])
def test_quant_pack_ragged(N, T, E, R, H):
    w = W.Workload("q", N=N, T=T, E=E, R=R, H=H, seed=N * T)
    _run(w, W.make_inputs(w))


def test_quant_pack_zero_blocks_tiny_values_and_signed_zeros():
    w = W.Workload("qz", N=2, T=64, E=8, R=2, H=512, seed=31)
    inp = W.make_inputs(w)
    x = inp.x.to(torch.float32)
    x[:, 0:128] = 0.0                       # all-zero block: scale 0, codes 0
    x[::2, 128:256] *= 1e-30                # tiny values (still bf16 normals/subnormals)
    x[1::2, 256:384] = -0.0                 # negative zeros next to normal values
    x[1::2, 300] = 3.0
    x[:, 384] = 1e-6                        # underflows to a zero code after scaling
    x[:, 385] = -1e-6
    x[:, 386] = 50.0
    inp.x = x.to(torch.bfloat16)
    _run(w, inp)


# the decode-fused form (moe_dispatch_fused_quant): the same checks plus its
# routing and counts against the oracle
@pytest.mark.parametrize("name", ["dsv3_decode", "kimi_k2_decode"])
def test_fused_quant_full_size(name):
    w = W.WORKLOADS[name]
    _run(w, W.make_inputs(w), fused=True)


@pytest.mark.parametrize("N,T,E,R,H", [(3, 77, 24, 3, 128), (4, 50, 32, 5, 384),
                                       (2, 300, 16, 2, 1152), (2, 24, 8, 3, 36864),
                                       (124, 33, 496, 8, 128)])
def test_fused_quant_ragged(N, T, E, R, H):
    w = W.Workload("fq", N=N, T=T, E=E, R=R, H=H, score_fn=W.SIGMOID, bias="normal",
                   renormalize=True, seed=N + T)
    _run(w, W.make_inputs(w), fused=True)


def test_fused_quant_rejects_other_rows_and_non_decode_batches():
    w = W.Workload("fqx", N=2, T=64, E=8, R=2, H=256, x_dtype=W.F32, seed=1)
    dims = moe.dims_of(w)
    b = moe.Buffers(dims)
    inp = W.make_inputs(w, device="cuda")
    q = moe.buffer_sizes(moe.fp8_dims(dims))
    pq = torch.empty(q["packed_x_bytes"], dtype=torch.uint8, device="cuda")
    ps = torch.empty(q["packed_scales_bytes"] // 4, dtype=torch.float32, device="cuda")
    ws = torch.zeros(max(16, b.sizes["fused_workspace_bytes"]), dtype=torch.uint8, device="cuda")
    with pytest.raises((moe.MoeError, ValueError)):  # f32 rows: the binding or the library refuses
        moe.dispatch_fused_quant(dims, inp.logits, None, w.score_fn, False, inp.x, b.topk_idx, b.topk_w,
                                 b.expert_counts, b.expert_offsets, b.rank_counts, b.rank_offsets,
                                 b.send_counts, b.pos, b.status, pq, ps, b.packed_src, ws)


def _quant_dispatch(w, inp, fused):
    """Every output of the fp8 dispatch, as the three calls or as one."""
    dims = moe.dims_of(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    b = moe.Buffers(dims, device=dev)
    q = moe.buffer_sizes(moe.fp8_dims(dims))
    pq = torch.zeros(q["packed_x_bytes"], dtype=torch.uint8, device=dev)
    ps = torch.zeros(q["packed_scales_bytes"] // 4, dtype=torch.float32, device=dev)
    for t in (b.topk_idx, b.topk_w, b.expert_counts, b.expert_offsets, b.rank_counts, b.rank_offsets,
              b.send_counts, b.pos, b.status, b.packed_src):
        t.view(torch.uint8).zero_()
    logits, x = inp.logits.to(dev), inp.x.to(dev)
    bias = None if inp.bias is None else inp.bias.to(dev)
    if fused:
        ws = torch.zeros(b.sizes["fused_workspace_bytes"], dtype=torch.uint8, device=dev)
        moe.dispatch_fused_quant(dims, logits, bias, w.score_fn, w.renormalize, x, b.topk_idx, b.topk_w,
                                 b.expert_counts, b.expert_offsets, b.rank_counts, b.rank_offsets,
                                 b.send_counts, b.pos, b.status, pq, ps, b.packed_src, ws)
    else:
        moe.route_topk(dims, logits, bias, w.score_fn, w.renormalize, b.topk_idx, b.topk_w)
        moe.dispatch_count(dims, b.topk_idx, b.expert_counts, b.expert_offsets, b.rank_counts,
                           b.rank_offsets, b.send_counts, b.pos, b.status)
        moe.dispatch_pack_quant(dims, x, b.pos, pq, ps, b.packed_src)
    torch.cuda.synchronize()
    out = {k: getattr(b, k).cpu().numpy() for k in ("topk_idx", "topk_w", "expert_counts", "expert_offsets",
                                                     "rank_counts", "rank_offsets", "send_counts", "pos",
                                                     "status", "packed_src")}
    out["packed_q"] = pq.cpu().numpy()
    out["packed_scales"] = ps.cpu().numpy().view(np.uint32)
    return out


@pytest.mark.parametrize("w", [
    # capacity overflow: rows past a rank's 300 are dropped (pos = -1)
    W.Workload("fq_cap", N=8, T=96, E=32, R=4, H=256, cap_rows=300, seed=201),
    # the DeepSeek-V3 convention of the bias (selection only)
    W.Workload("fq_bsel", N=16, T=64, E=256, R=8, H=384, score_fn=W.SIGMOID | moe.MOE_BIAS_SELECT_ONLY,
               bias="normal", renormalize=True, seed=202),
], ids=lambda w: w.name)
def test_fused_quant_equals_the_three_calls_bytewise(w):
    inp = W.make_inputs(w)
    a = _quant_dispatch(w, inp, fused=True)
    b = _quant_dispatch(w, inp, fused=False)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    if w.name == "fq_cap":
        assert int(a["status"][0]) == moe.MOE_ERR_CAPACITY
