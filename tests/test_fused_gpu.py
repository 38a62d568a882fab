"""Parity of the decode-fused dispatch (route + count + pack in one call:
one thread-block cluster for small batches, else a route kernel that also
counts, whose last block scans the counts, followed by a pack kernel that
derives the rows itself) with the oracle; same bar as the separate calls: indices, counts, positions
and packed rows bit-exact (and nothing written outside the occupied rows),
weights within 2e-6, combine within the combine tolerance."""
import numpy as np
import pytest
import torch

import combine_moe_route_topk_gb300 as moe
import oracle
from combine_moe_route_topk_gb300 import workloads as W
from gpu_path import GpuRun
from test_parity_gpu import _compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "kimi_k2_decode"])
def test_fused_full_size_decode(name):
    w = W.WORKLOADS[name]
    gr, _, _ = _compare(w, W.make_inputs(w), fused=True)
    assert gr.status == oracle.OK


CASES = {
    # ties, sigmoid without renormalisation, a bias
    "ties_sigmoid": W.Workload("ties_sigmoid", N=8, T=32, E=64, R=6, H=256, score_fn=W.SIGMOID,
                               bias="normal", seed=61),
    # one expert per rank, f32 rows, N*T = 672 split unevenly over the blocks
    "f32_ragged": W.Workload("f32_ragged", N=7, T=96, E=14, R=2, H=72, x_dtype=W.F32,
                             y_dtype=W.F32, renormalize=True, seed=62),
    # fp8 rows with block scales (512 tokens: the single-cluster path)
    "fp8": W.Workload("fp8", N=8, T=64, E=64, R=4, H=512, x_dtype=W.FP8E4M3_BLK128,
                      expert_op=W.EXPERT_DEQUANT, seed=63),
    # fp8 rows with block scales through the two-kernel form (1536 tokens,
    # three route blocks per source rank)
    "fp8_two_kernel": W.Workload("fp8_two_kernel", N=16, T=96, E=128, R=8, H=1024,
                                 x_dtype=W.FP8E4M3_BLK128, expert_op=W.EXPERT_DEQUANT,
                                 renormalize=True, seed=83),
    # more experts per lane (E = 512)
    "e512": W.Workload("e512", N=16, T=64, E=512, R=8, H=128, renormalize=True, seed=64),
    # capacity overflow reported through the status word
    "capacity": W.Workload("capacity", N=4, T=64, E=16, R=2, H=128, cap_rows=100, seed=65),
    # the largest batch the single-cluster path takes: 16 blocks of 32 tokens,
    # E = 256, R = 8 (rows of 512 bytes: 147 KB read and written per block)
    "small_max": W.Workload("small_max", N=16, T=32, E=256, R=8, H=256, score_fn=W.SIGMOID,
                            renormalize=True, bias="normal", seed=66),
    # odd E: the single-cluster path (64 tokens) and the two-kernel form (960 tokens)
    "odd_e_small": W.Workload("odd_e_small", N=1, T=64, E=7, R=3, H=64, seed=69),
    "odd_e_two_kernel": W.Workload("odd_e_two_kernel", N=3, T=320, E=9, R=3, H=64, seed=70),
    # 256 tokens with 14 KB rows: too much row traffic for the cluster path
    "wide_rows_256": W.Workload("wide_rows_256", N=2, T=128, E=16, R=4, H=7168,
                                score_fn=W.SIGMOID, renormalize=True, bias="normal",
                                expert_op=W.EXPERT_SCALE, seed=71),
    # T not a multiple of 32: four blocks per source rank, the last with 4 tokens
    "t100": W.Workload("t100", N=8, T=100, E=64, R=6, H=256, renormalize=True,
                       bias="normal", seed=74),
    # R = 16 (512 pairs in a block of 32 tokens)
    "r16": W.Workload("r16", N=4, T=160, E=64, R=16, H=128, score_fn=W.SIGMOID, seed=75),
    # R = 32: 1024 pairs, one per thread of a route block
    "r32": W.Workload("r32", N=4, T=192, E=64, R=32, H=64, renormalize=True, seed=79),
    # one token per rank and 512 ranks: blocks of 32 whole source ranks
    "t1_n512": W.Workload("t1_n512", N=512, T=1, E=512, R=4, H=64, bias="normal", seed=76),
    # T = 5: six whole source ranks per block, the last block with two
    "t5_n200": W.Workload("t5_n200", N=200, T=5, E=400, R=4, H=64, renormalize=True, seed=80),
    # T = 17: one whole source rank per block, 17 tokens each
    "t17": W.Workload("t17", N=48, T=17, E=96, R=5, H=64, score_fn=W.SIGMOID, seed=81),
    # T = 33: two blocks per source rank, the second with one token; the
    # largest workspace of the fused form (248 route blocks, E = 496)
    "t33_n124_e496": W.Workload("t33_n124_e496", N=124, T=33, E=496, R=8, H=64, renormalize=True,
                                seed=82),
    # the largest batch with the widest expert table (4096 tokens, E = 512:
    # 16 experts per lane)
    "n4096_e512": W.Workload("n4096_e512", N=16, T=256, E=512, R=8, H=256,
                             score_fn=W.SIGMOID, renormalize=True, bias="normal", seed=77),
    # a single route block, which is also the one that scans (32 tokens of
    # one rank with 14 KB rows: past the cluster path's row traffic)
    "one_route_block": W.Workload("one_route_block", N=1, T=32, E=16, R=4, H=7168, score_fn=W.SIGMOID,
                                  renormalize=True, bias="normal", seed=84),
    # capacity overflow
    "capacity_two_kernel": W.Workload("capacity_two_kernel", N=8, T=96, E=32, R=4, H=128,
                                      cap_rows=300, seed=78),
    # shapes only the single-cluster path takes: one token per rank (T % 32
    # != 0) and R > 8
    "decode_t1": W.Workload("decode_t1", N=64, T=1, E=128, R=8, H=256, score_fn=W.SIGMOID,
                            renormalize=True, bias="normal", seed=72),
    "r12_t24": W.Workload("r12_t24", N=8, T=24, E=64, R=12, H=128, renormalize=True, seed=73),
    # a cluster of one block: one rank, 32 tokens
    "one_block": W.Workload("one_block", N=1, T=32, E=8, R=2, H=64, bias="normal", seed=68),
    # past the cluster path's per-block row traffic (1.2 MB of 256 KB): two-kernel form
    "past_small": W.Workload("past_small", N=16, T=32, E=256, R=8, H=2048, score_fn=W.SIGMOID,
                             renormalize=True, bias="normal", seed=67),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fused_cases(name):
    w = CASES[name]
    inp = W.make_inputs(w, tie_every=3 if name == "ties_sigmoid" else 0)
    gr, _, _ = _compare(w, inp, fused=True)
    assert gr.status == (oracle.ERR_CAPACITY if name in ("capacity", "capacity_two_kernel") else oracle.OK)


# dsv3_decode, kimi_k2_decode, past_small, t100, r16, r32, t1_n512, t5_n200,
# t33_n124_e496, fp8_two_kernel and one_route_block take the two-kernel form; tiny, small_max, decode_t1 and
# r12_t24 the single thread-block cluster (up to 512 tokens, E <= 256, at most
# 256 KB of rows read and written per 32 tokens)
@pytest.mark.parametrize("name", ["dsv3_decode", "kimi_k2_decode", "past_small", "tiny", "small_max",
                                  "decode_t1", "r12_t24", "t100", "r16", "r32", "t1_n512", "t5_n200",
                                  "t33_n124_e496", "fp8_two_kernel", "one_route_block"])
def test_fused_equals_separate_calls_bytewise(name):
    w = W.WORKLOADS.get(name) or CASES[name]
    inp = W.make_inputs(w)
    a = GpuRun(w, inp, fused=True)
    b = GpuRun(w, inp)
    for k in a.host:
        np.testing.assert_array_equal(a.host[k], b.host[k], err_msg=k)
    pa, sca, sa = a.packed_rows()
    pb, scb, sb = b.packed_rows()
    np.testing.assert_array_equal(pa, pb)
    np.testing.assert_array_equal(sa, sb)
    if sca is not None or scb is not None:  # fp8 rows: the block scales too
        np.testing.assert_array_equal(sca, scb)


@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("E", [32, 1024])  # E = 1024 is past both fused forms' limits
def test_fused_empty_batch(static, E):
    """N*T == 0 is always accepted: zero counts and offsets, MOE_OK, as the
    separate calls give."""
    w = W.Workload("empty", N=4, T=0, E=E, R=17, H=64)
    dims = moe.dims_of(w)
    b = moe.Buffers(dims)
    for t in (b.expert_counts, b.expert_offsets, b.rank_counts, b.rank_offsets, b.send_counts):
        t.fill_(7)
    b.status.fill_(-99)
    x = torch.empty(0, w.H, dtype=torch.bfloat16, device="cuda")
    logits = torch.empty(0, w.E, dtype=torch.float32, device="cuda")
    args = (dims, logits, None, W.SOFTMAX, False, x, None, b.topk_idx, b.topk_w, b.expert_counts,
            b.expert_offsets, b.rank_counts, b.rank_offsets, b.send_counts, b.pos, b.status,
            b.packed_x, None, b.packed_src)
    if static:
        moe.dispatch_fused_static(*args)
    else:
        # an empty batch touches no workspace: none is passed
        assert moe.buffer_sizes(dims)["fused_workspace_bytes"] == 0
        moe.dispatch_fused(*args, None)
    assert moe.read_status(b.status) == moe.MOE_OK
    for t in (b.expert_counts, b.expert_offsets, b.rank_counts, b.rank_offsets, b.send_counts):
        assert int(t.abs().sum()) == 0


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode"])
def test_fused_dispatch_captures_into_a_cuda_graph(name):
    """moe_dispatch_fused enqueues only kernels with fixed shapes (the
    single-cluster kernel, or the route kernel that counts and the pack
    kernel), so it captures into a CUDA graph; a replay on new
    inputs gives the oracle's routing, counts, positions and rows."""
    w = W.WORKLOADS[name]
    dims = moe.dims_of(w)
    b = moe.Buffers(dims)
    inp = W.make_inputs(w, device="cuda")
    logits, x = inp.logits.clone(), inp.x.clone()
    bias = None if inp.bias is None else inp.bias.clone()
    ws = torch.zeros(b.sizes["fused_workspace_bytes"], dtype=torch.uint8, device="cuda")

    def call():
        moe.dispatch_fused(dims, logits, bias, w.score_fn, w.renormalize, x, None, b.topk_idx,
                           b.topk_w, b.expert_counts, b.expert_offsets, b.rank_counts,
                           b.rank_offsets, b.send_counts, b.pos, b.status, b.packed_x, None,
                           b.packed_src, ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # warm-up outside the capture (sets kernel attributes)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    w2 = w.replace(seed=w.seed + 7)
    inp2 = W.make_inputs(w2)
    logits.copy_(inp2.logits)
    x.copy_(inp2.x)
    if bias is not None:
        bias.copy_(inp2.bias)
    b.pos.fill_(-5)
    graph.replay()
    torch.cuda.synchronize()
    assert moe.read_status(b.status) == moe.MOE_OK
    ref = oracle.run(w2, inp2, with_combine=False)
    np.testing.assert_array_equal(b.topk_idx.cpu().numpy(), ref["topk_idx"])
    np.testing.assert_allclose(b.topk_w.cpu().numpy(), ref["topk_w"], rtol=2e-6, atol=0)
    for k in ("expert_counts", "expert_offsets", "rank_counts", "rank_offsets", "send_counts", "pos"):
        np.testing.assert_array_equal(getattr(b, k).cpu().numpy(), ref[k], err_msg=k)
    pos = ref["pos"].ravel()
    pos = pos[pos >= 0]
    crow = ref["rank_offsets"][pos // ref["cap"]] + pos % ref["cap"]
    got = oracle.x_as_bytes(b.packed_x[torch.from_numpy(pos).long().cuda()].cpu())
    np.testing.assert_array_equal(got, ref["packed_x"][crow])


@pytest.mark.parametrize("name", ["dsv3_decode", "t33_n124_e496", "t5_n200"])
def test_fused_call_leaves_the_workspace_ready_for_the_next(name):
    """The two-kernel form requires a workspace whose arrival counter (its
    first word) is zero; every call must leave it so.  A second call on the
    same workspace then gives the same outputs as the first."""
    w = W.WORKLOADS.get(name) or CASES[name]
    inp = W.make_inputs(w)
    dims = moe.dims_of(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    d = W.Inputs(*(t.to(dev) if t is not None else None for t in (inp.logits, inp.bias, inp.x, inp.x_scales)))
    b = moe.Buffers(dims, device=dev)
    ws = torch.zeros(b.sizes["fused_workspace_bytes"], dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(2):
        moe.dispatch_fused(dims, d.logits, d.bias, w.score_fn, w.renormalize, d.x, d.x_scales, b.topk_idx,
                           b.topk_w, b.expert_counts, b.expert_offsets, b.rank_counts, b.rank_offsets,
                           b.send_counts, b.pos, b.status, b.packed_x, b.packed_scales, b.packed_src, ws)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32)[0]) == 0
        outs.append({k: getattr(b, k).clone() for k in ("topk_idx", "expert_offsets", "send_counts", "pos")})
    for k in outs[0]:
        assert torch.equal(outs[0][k], outs[1][k]), k
