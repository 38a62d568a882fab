"""Route top-k with the bias in the selection key only (score_fn |
MOE_BIAS_SELECT_ONLY, the DeepSeek-V3 router convention) against the oracle.

Both sides decide the selection on float32 keys fl32(s + bias), s being the
score of the raw logit.  The oracle's s is the float32 rounding of its fp64
score; the kernel computes s in float32 (expf within 2 ulp, one addition,
one division), so the two can differ by a few ulp and keys that close may
order differently.  The bar:

* a token whose selection equals the oracle's must have weights within the
  relative 2e-6 of the other route tests;
* any other token must be a near-tie: its selection is a valid top-R, in
  order, of the keys recomputed here in fp64 from the raw scores, up to an
  absolute slack of 1e-6 (scores lie in [0, 1], so a few ulp of s plus one
  rounding of a key of magnitude < 4 stays below 5e-7), and its weights are
  the raw scores of its own selection.  Such tokens are rare: two selected
  (or boundary) experts whose raw scores lie within a few ulp of each other,
  e.g. logits 1.9048145 and 1.9048139 under a softmax over 256 experts, about
  one token in ten thousand.  Their number is capped at max(2, N*T/1000) only
  as a guard against a systematic error, which the near-tie check below
  would catch as well.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_topk_gb300 as moe
import oracle
from combine_moe_route_topk_gb300 import workloads as W
from gpu_path import GpuRun, TOPK_W_RTOL
from test_parity_gpu import _compare

pytestmark = pytest.mark.gpu

FLAG = moe.MOE_BIAS_SELECT_ONLY
KEY_SLACK = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()


def _raw_scores64(logits: np.ndarray, softmax: bool) -> np.ndarray:
    l = logits.astype(np.float64)
    if softmax:
        e = np.exp(l - l.max(axis=1, keepdims=True))
        return e / e.sum(axis=1, keepdims=True)
    return 1.0 / (1.0 + np.exp(-l))


def _check_route(w: W.Workload, inp: W.Inputs):
    dims = moe.dims_of(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    logits_d = inp.logits.to(dev)
    bias_d = None if inp.bias is None else inp.bias.to(dev)
    idx_d = torch.empty(w.NT, w.R, dtype=torch.int32, device=dev)
    w_d = torch.empty(w.NT, w.R, dtype=torch.float32, device=dev)
    moe.route_topk(dims, logits_d, bias_d, w.score_fn, w.renormalize, idx_d, w_d)
    torch.cuda.synchronize()
    gi, gw = idx_d.cpu().numpy(), w_d.cpu().numpy()

    logits = inp.logits.numpy()
    bias = None if inp.bias is None else inp.bias.numpy()
    oi, ow, _ = oracle.route(logits, bias, w.R, w.score_fn, w.renormalize)
    same = (gi == oi).all(axis=1)
    np.testing.assert_allclose(gw[same], ow[same], rtol=TOPK_W_RTOL, atol=0)
    diff = np.flatnonzero(~same)
    assert len(diff) <= max(2, w.NT // 1000), f"{len(diff)} tokens select differently from the oracle"
    if len(diff) == 0:
        return
    s64 = _raw_scores64(logits[diff], (w.score_fn & ~FLAG) == W.SOFTMAX)
    keys = s64 + (0.0 if bias is None else bias.astype(np.float64))
    for row, g in enumerate(diff):
        sel = gi[g].astype(np.int64)
        assert len(set(sel.tolist())) == w.R and sel.min() >= 0 and sel.max() < w.E
        k_sel = keys[row, sel]
        rest = np.ones(w.E, bool)
        rest[sel] = False
        assert k_sel.min() >= keys[row, rest].max() - KEY_SLACK, f"token {g}: not a near-tie"
        assert np.all(np.diff(k_sel) <= KEY_SLACK), f"token {g}: order"
        want = s64[row, sel]
        if w.renormalize:
            want = want / want.sum()
        np.testing.assert_allclose(gw[g], want, rtol=TOPK_W_RTOL, atol=0)


CASES = {
    "tiny_softmax_bias": (W.WORKLOADS["tiny"].replace(bias="normal", score_fn=W.SOFTMAX | FLAG), 3),
    # equal logits give bit-identical scores on both sides: ties to the lower index
    "tiny_sigmoid_ties": (W.WORKLOADS["tiny"].replace(score_fn=W.SIGMOID | FLAG, renormalize=True), 2),
    "dsv3_decode": (W.WORKLOADS["dsv3_decode"].replace(score_fn=W.SIGMOID | FLAG), 0),
    "kimi_k2_decode": (W.WORKLOADS["kimi_k2_decode"].replace(score_fn=W.SOFTMAX | FLAG), 0),
    "qwen3_235b_prefill": (W.WORKLOADS["qwen3_235b_prefill"].replace(score_fn=W.SOFTMAX | FLAG), 0),
    "skewed": (W.WORKLOADS["skewed"].replace(score_fn=W.SOFTMAX | FLAG), 0),
    # E % 4 != 0 (scalar loads), ragged last lane
    "e37_scalar": (W.Workload("e37", N=1, T=97, E=37, R=5, H=8, bias="normal",
                              score_fn=W.SIGMOID | FLAG, seed=71), 4),
    # 32 experts per lane
    "e1024": (W.Workload("e1024", N=16, T=64, E=1024, R=8, H=8, bias="normal",
                         score_fn=W.SOFTMAX | FLAG, renormalize=True, seed=72), 0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_route_bias_select_only(name):
    w, tie_every = CASES[name]
    _check_route(w, W.make_inputs(w, tie_every=tie_every))


def test_saturated_sigmoid_scores_tie_to_the_lower_index():
    # logits of 20 and above give a float score of exactly 1 on both sides
    w = W.Workload("sat", N=2, T=64, E=32, R=4, H=8, score_fn=W.SIGMOID | FLAG, seed=73)
    inp = W.make_inputs(w)
    inp.logits[:, 5] = 20.0
    inp.logits[:, 9] = 30.0
    inp.logits[:, 20] = 25.0
    _check_route(w, inp)
    idx, _, _ = oracle.route(inp.logits.numpy(), None, 4, w.score_fn, False)
    assert (idx[:, :3] == [5, 9, 20]).all()


def test_bias_select_full_path_small():
    # route -> count -> pack -> combine with the flag; a small batch has no
    # near-ties, so every output matches the oracle at the usual bar
    w = W.WORKLOADS["tiny"].replace(bias="normal", score_fn=W.SIGMOID | FLAG, renormalize=True)
    _compare(w, W.make_inputs(w))
    _compare(w, W.make_inputs(w), fused=True)


NEAR_TIE_ULPS = 64


def _without_near_ties(w: W.Workload, inp: W.Inputs) -> W.Inputs:
    """The same inputs with every near-tie token (two of its R+1 highest keys,
    recomputed here in fp64 from the raw scores and rounded scores, less than
    NEAR_TIE_ULPS units in the last place apart) given the logits of a token
    far from any tie.  On such an input any f32 evaluation of the keys makes
    the oracle's selection, so count, pack and combine can be compared with
    it at the usual bar.  The DeepSeek-V3-shaped batch (seed 0) has four such
    tokens of 4096, the Kimi-K2-shaped one three."""
    logits = inp.logits.numpy().astype(np.float64)
    s = _raw_scores64(logits, (w.score_fn & ~FLAG) == W.SOFTMAX).astype(np.float32)
    keys = s.astype(np.float64) + (0.0 if inp.bias is None else inp.bias.numpy().astype(np.float64))
    top = -np.sort(-keys, axis=1)[:, :w.R + 1]
    ulp = np.spacing(np.abs(top).max(axis=1).astype(np.float32)).astype(np.float64)
    near = np.diff(-top, axis=1).min(axis=1) < NEAR_TIE_ULPS * ulp
    far = np.flatnonzero(~near)
    assert far.size > 0 and near.sum() <= w.NT // 100
    out = W.Inputs(inp.logits.clone(), inp.bias, inp.x, inp.x_scales)
    if near.any():
        out.logits[torch.from_numpy(np.flatnonzero(near))] = inp.logits[int(far[0])]
    return out


@pytest.mark.parametrize("name", ["dsv3_decode", "kimi_k2_decode"])
def test_bias_select_full_path_full_size(name):
    """Route -> count -> pack -> combine with the flag at full size, every
    output against the oracle (and nothing written outside the occupied
    rows), on the workload's inputs with its near-tie tokens replaced."""
    base = W.WORKLOADS[name]
    fn = (base.score_fn & ~FLAG) | FLAG
    w = base.replace(score_fn=fn)
    _compare(w, _without_near_ties(w, W.make_inputs(w)))


def test_bias_select_fused_equals_separate_calls():
    w = W.WORKLOADS["dsv3_decode"].replace(score_fn=W.SIGMOID | FLAG)
    inp = W.make_inputs(w)
    a = GpuRun(w, inp, fused=True)
    b = GpuRun(w, inp)
    for k in a.host:
        np.testing.assert_array_equal(a.host[k], b.host[k], err_msg=k)
