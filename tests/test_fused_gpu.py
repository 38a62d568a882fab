"""Parity of the decode-fused dispatch (route + count + pack in one launch:
one thread-block cluster for small batches, else one cooperative launch)
with the oracle; same bar as the separate calls: indices, counts, positions
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
    # fp8 rows with block scales
    "fp8": W.Workload("fp8", N=8, T=64, E=64, R=4, H=512, x_dtype=W.FP8E4M3_BLK128,
                      expert_op=W.EXPERT_DEQUANT, seed=63),
    # more experts per lane (E = 512)
    "e512": W.Workload("e512", N=16, T=64, E=512, R=8, H=128, renormalize=True, seed=64),
    # capacity overflow reported through the status word
    "capacity": W.Workload("capacity", N=4, T=64, E=16, R=2, H=128, cap_rows=100, seed=65),
    # the largest batch the single-cluster path takes: 16 blocks of 32 tokens,
    # E = 256, R = 8 (rows of 512 bytes: 147 KB read and written per block)
    "small_max": W.Workload("small_max", N=16, T=32, E=256, R=8, H=256, score_fn=W.SIGMOID,
                            renormalize=True, bias="normal", seed=66),
    # odd E: the single-cluster path (64 tokens) and the cooperative kernel (960 tokens)
    "odd_e_small": W.Workload("odd_e_small", N=1, T=64, E=7, R=3, H=64, seed=69),
    "odd_e_coop": W.Workload("odd_e_coop", N=3, T=320, E=9, R=3, H=64, seed=70),
    # 256 tokens with 14 KB rows: too much row traffic for the cluster path, so
    # the cooperative kernel runs with one token per block
    "coop_one_token_blocks": W.Workload("coop_one_token_blocks", N=2, T=128, E=16, R=4, H=7168,
                                        score_fn=W.SIGMOID, renormalize=True, bias="normal",
                                        expert_op=W.EXPERT_SCALE, seed=71),
    # cooperative kernel, T not a multiple of 32 (blocks straddle source ranks)
    "coop_t100": W.Workload("coop_t100", N=8, T=100, E=64, R=6, H=256, renormalize=True,
                            bias="normal", seed=74),
    # cooperative kernel, R = 16 (512 pairs in a block of 32 tokens at most)
    "coop_r16": W.Workload("coop_r16", N=4, T=160, E=64, R=16, H=128, score_fn=W.SIGMOID, seed=75),
    # cooperative kernel, one token per rank and 512 ranks: blocks of one or
    # two tokens, each from its own source rank
    "coop_t1_n512": W.Workload("coop_t1_n512", N=512, T=1, E=512, R=4, H=64, bias="normal",
                               seed=76),
    # cooperative kernel at its largest batch with the widest expert table
    # (4096 tokens, E = 512: 16 experts per lane)
    "coop_4096_e512": W.Workload("coop_4096_e512", N=16, T=256, E=512, R=8, H=256,
                                 score_fn=W.SIGMOID, renormalize=True, bias="normal", seed=77),
    # cooperative kernel, capacity overflow
    "coop_capacity": W.Workload("coop_capacity", N=8, T=96, E=32, R=4, H=128, cap_rows=300,
                                seed=78),
    # shapes only the single-cluster path takes: one token per rank (T % 32
    # != 0) and R > 8
    "decode_t1": W.Workload("decode_t1", N=64, T=1, E=128, R=8, H=256, score_fn=W.SIGMOID,
                            renormalize=True, bias="normal", seed=72),
    "r12_t24": W.Workload("r12_t24", N=8, T=24, E=64, R=12, H=128, renormalize=True, seed=73),
    # a cluster of one block: one rank, 32 tokens
    "one_block": W.Workload("one_block", N=1, T=32, E=8, R=2, H=64, bias="normal", seed=68),
    # past the cluster path's per-block row traffic (1.2 MB): cooperative kernel
    "past_small": W.Workload("past_small", N=16, T=32, E=256, R=8, H=2048, score_fn=W.SIGMOID,
                             renormalize=True, bias="normal", seed=67),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fused_cases(name):
    w = CASES[name]
    inp = W.make_inputs(w, tie_every=3 if name == "ties_sigmoid" else 0)
    gr, _, _ = _compare(w, inp, fused=True)
    assert gr.status == (oracle.ERR_CAPACITY if name in ("capacity", "coop_capacity") else oracle.OK)


# dsv3_decode, kimi_k2_decode, past_small and the coop_ cases take the
# cooperative kernel; tiny and small_max the single thread-block cluster (up
# to 512 tokens, E <= 256, at most 1 MB of rows read and written per 32 tokens)
@pytest.mark.parametrize("name", ["dsv3_decode", "kimi_k2_decode", "past_small", "tiny", "small_max",
                                  "decode_t1", "r12_t24", "coop_t100", "coop_r16", "coop_t1_n512"])
def test_fused_equals_separate_calls_bytewise(name):
    w = W.WORKLOADS.get(name) or CASES[name]
    inp = W.make_inputs(w)
    a = GpuRun(w, inp, fused=True)
    b = GpuRun(w, inp)
    for k in a.host:
        np.testing.assert_array_equal(a.host[k], b.host[k], err_msg=k)
    pa, _, sa = a.packed_rows()
    pb, _, sb = b.packed_rows()
    np.testing.assert_array_equal(pa, pb)
    np.testing.assert_array_equal(sa, sb)


@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("R", [2, 17])  # R = 17 is past both fused kernels' limits
def test_fused_empty_batch(static, R):
    """N*T == 0 is always accepted: zero counts and offsets, MOE_OK, as the
    separate calls give."""
    w = W.Workload("empty", N=4, T=0, E=32, R=R, H=64)
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
        ws = torch.empty(moe.buffer_sizes(dims)["fused_workspace_bytes"], dtype=torch.uint8,
                         device="cuda")
        moe.dispatch_fused(*args, ws)
    assert moe.read_status(b.status) == moe.MOE_OK
    for t in (b.expert_counts, b.expert_offsets, b.rank_counts, b.rank_offsets, b.send_counts):
        assert int(t.abs().sum()) == 0


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode"])
def test_fused_dispatch_captures_into_a_cuda_graph(name):
    """moe_dispatch_fused enqueues only stream work with fixed shapes (the
    single-cluster kernel, or a memset, the cooperative route-count kernel
    and the pack kernel), so it captures into a CUDA graph; a replay on new
    inputs gives the oracle's routing, counts, positions and rows."""
    w = W.WORKLOADS[name]
    dims = moe.dims_of(w)
    b = moe.Buffers(dims)
    inp = W.make_inputs(w, device="cuda")
    logits, x = inp.logits.clone(), inp.x.clone()
    bias = None if inp.bias is None else inp.bias.clone()
    ws = torch.empty(b.sizes["fused_workspace_bytes"], dtype=torch.uint8, device="cuda")

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
