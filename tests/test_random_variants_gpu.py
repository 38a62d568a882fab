"""Seeded sweeps of random shapes through the other entry points, each at the
bar of its own tests:

* decode-fused dispatch (both the single-cluster and the two-kernel form)
  against the three separate calls, byte for byte;
* the quantising pack against the oracle (codes and scales bit-exact), also
  through the decode-fused fp8 dispatch (routing and counts too);
* the expert-parallel local path of a rank and the send-side partials
  against the oracle;
* the bias-for-selection-only router against the oracle (near-tie rule).

Shapes vary ranks, experts per rank (odd counts included), R, tokens per
rank, row widths and dtypes, score function, bias, renormalisation and
capacity."""
import random

import numpy as np
import pytest

import combine_moe_route_topk_gb300 as moe
from combine_moe_route_topk_gb300 import workloads as W
from gpu_path import GpuRun
import sweep_params as S
from test_pack_quant_gpu import _run as run_quant
from test_rank_partials_gpu import (check_local_accumulation, check_pack_rank,
                                    check_send_side_partials)
from test_route_bias_select_gpu import _check_route

pytestmark = pytest.mark.gpu

FLAG = moe.MOE_BIAS_SELECT_ONLY


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()


def _rows(rng, allow_fp8=True):
    x_dtype = rng.choice([W.BF16, W.BF16, W.F32] + ([W.FP8E4M3_BLK128] if allow_fp8 else []))
    if x_dtype == W.FP8E4M3_BLK128:
        return x_dtype, 128 * rng.randint(1, 3), W.BF16, W.EXPERT_DEQUANT
    y_dtype = rng.choice([x_dtype, W.F32 if x_dtype == W.BF16 else W.BF16])
    return x_dtype, 8 * rng.randint(1, 96), y_dtype, rng.choice([W.EXPERT_IDENTITY, W.EXPERT_SCALE])


def _fused_shapes(n, seed=31):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.choice([1, 2, 3, 4, 8, 16, 32, 64, 128])
        E = N * rng.choice([1, 2, 3, 5, 8, 16, 32])
        while E > 512:
            E //= 2
        E = max(N, E // N * N)
        R = rng.randint(1, min(E, 32))
        T = rng.randint(1, max(1, min(256, 4096 // N)))
        x_dtype, H, y_dtype, op = _rows(rng)
        score = rng.choice([W.SOFTMAX, W.SIGMOID]) | (FLAG if rng.random() < 0.25 else 0)
        cap = 0 if rng.random() < 0.8 else max(1, N * T * max(R, E // N) // 16)
        out.append(W.Workload(f"fused{i}", N=N, T=T, E=E, R=R, H=H, x_dtype=x_dtype, y_dtype=y_dtype,
                              expert_op=op, score_fn=score, renormalize=rng.random() < 0.5,
                              bias=rng.choice(["none", "normal"]), cap_rows=cap, seed=2000 + i))
    return out


def _small_fused_shapes(n, seed=33):
    """Batches only the single-cluster path takes: any T, R up to 32."""
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.choice([1, 2, 4, 8, 16, 64])
        E = N * rng.choice([1, 2, 3, 4])
        while E > 256:
            E //= 2
        E = max(N, E // N * N)
        R = rng.randint(1, min(E, 32))
        T = rng.randint(1, max(1, 512 // N))
        x_dtype, H, y_dtype, op = _rows(rng)
        if x_dtype == W.FP8E4M3_BLK128:
            H = 128
        else:
            # keep the rows within the cluster path's traffic limit: 32 tokens
            # x (1 + R) rows of at most 256 KB per block
            elem = 4 if x_dtype == W.F32 else 2
            H = max(8, min(H, 256, (256 << 10) // (32 * (R + 1) * elem) // 8 * 8))
        out.append(W.Workload(f"small{i}", N=N, T=T, E=E, R=R, H=H, x_dtype=x_dtype, y_dtype=y_dtype,
                              expert_op=op, score_fn=rng.choice([W.SOFTMAX, W.SIGMOID]),
                              renormalize=rng.random() < 0.5, bias=rng.choice(["none", "normal"]),
                              seed=2500 + i))
    return out


@pytest.mark.parametrize("w", _fused_shapes(S.count(16), S.seed(31)) + _small_fused_shapes(S.count(12), S.seed(33)), ids=lambda w: w.name)
def test_random_fused_equals_separate_calls(w):
    inp = W.make_inputs(w)
    try:
        a = GpuRun(w, inp, fused=True)
    except moe.MoeError as ex:
        if ex.code == moe.MOE_ERR_UNSUPPORTED:
            pytest.skip(str(ex))
        raise
    b = GpuRun(w, inp)
    assert a.status == b.status
    for k in a.host:
        np.testing.assert_array_equal(a.host[k], b.host[k], err_msg=k)
    pa, sca, sa = a.packed_rows()
    pb, scb, sb = b.packed_rows()
    np.testing.assert_array_equal(pa, pb)
    np.testing.assert_array_equal(sa, sb)
    if sca is not None:
        np.testing.assert_array_equal(sca, scb)


def _quant_shapes(n, seed=37):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.choice([1, 2, 3, 4, 8])
        E = N * rng.choice([1, 2, 3, 7, 16])
        R = rng.randint(1, min(E, 32))
        out.append(W.Workload(f"quant{i}", N=N, T=rng.choice([1, 13, 64, 200]), E=E, R=R,
                              H=128 * rng.randint(1, 12), score_fn=rng.choice([W.SOFTMAX, W.SIGMOID]),
                              renormalize=rng.random() < 0.5, seed=3000 + i))
    return out


@pytest.mark.parametrize("w", _quant_shapes(S.count(10), S.seed(37)), ids=lambda w: w.name)
def test_random_quant_pack(w):
    run_quant(w, W.make_inputs(w))


def _fused_quant_shapes(n, seed=39):
    """Decode batches for moe_dispatch_fused_quant: up to 4096 tokens, E up to
    512, any T and R, bf16 rows of 128-element blocks."""
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.choice([1, 2, 4, 8, 16, 32, 64])
        E = N * rng.choice([1, 2, 3, 5, 8])
        while E > 512:
            E //= 2
        E = max(N, E // N * N)
        R = rng.randint(1, min(E, 32))
        T = rng.randint(1, max(1, min(256, 4096 // N)))
        out.append(W.Workload(f"fquant{i}", N=N, T=T, E=E, R=R, H=128 * rng.randint(1, 8),
                              score_fn=rng.choice([W.SOFTMAX, W.SIGMOID]),
                              renormalize=rng.random() < 0.5, bias=rng.choice(["none", "normal"]),
                              seed=3500 + i))
    return out


@pytest.mark.parametrize("w", _fused_quant_shapes(S.count(10), S.seed(39)), ids=lambda w: w.name)
def test_random_fused_quant(w):
    # routing, counts, positions, codes, scales and rows against the oracle
    # (the default reading of the bias: selection on exact f32 keys, so the
    # indices are compared bit for bit)
    run_quant(w, W.make_inputs(w), fused=True)


def _rank_shapes(n, seed=41):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.choice([2, 3, 4, 5, 8])
        E = N * rng.choice([1, 2, 3, 5, 8])
        R = rng.randint(1, min(E, 16))
        x_dtype, H, y_dtype, op = _rows(rng)
        out.append(W.Workload(f"rank{i}", N=N, T=rng.choice([1, 9, 40, 130]), E=E, R=R, H=H,
                              x_dtype=x_dtype, y_dtype=y_dtype, expert_op=op,
                              score_fn=rng.choice([W.SOFTMAX, W.SIGMOID]),
                              renormalize=rng.random() < 0.5, bias=rng.choice(["none", "normal"]),
                              seed=4000 + i))
    return out


RANK_SHAPES = _rank_shapes(S.count(8), S.seed(41))


@pytest.mark.parametrize("w", RANK_SHAPES, ids=lambda w: w.name)
def test_random_pack_rank(w):
    check_pack_rank(w)


@pytest.mark.parametrize("w", RANK_SHAPES, ids=lambda w: w.name)
def test_random_local_accumulation(w):
    check_local_accumulation(w)


@pytest.mark.parametrize("w", RANK_SHAPES, ids=lambda w: w.name)
def test_random_send_side_partials(w):
    check_send_side_partials(w)


def _select_shapes(n, seed=43):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.choice([1, 2, 4, 8])
        E = N * rng.choice([1, 3, 8, 32, 64, 128])
        R = rng.randint(1, min(E, 32))
        out.append(W.Workload(f"sel{i}", N=N, T=rng.choice([1, 17, 64, 300]), E=E, R=R, H=8,
                              score_fn=rng.choice([W.SOFTMAX, W.SIGMOID]) | FLAG,
                              renormalize=rng.random() < 0.5, bias=rng.choice(["none", "normal"]),
                              seed=5000 + i))
    return out


@pytest.mark.parametrize("w", _select_shapes(S.count(10), S.seed(43)), ids=lambda w: w.name)
def test_random_bias_select_route(w):
    _check_route(w, W.make_inputs(w))
