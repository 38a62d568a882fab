"""A seeded sweep of random small shapes through the whole path (route,
count, pack, expert op, combine) against the oracle, at the bar of the other
parity tests: indices, counts, positions, packed rows and sources bit-exact,
weights within 2e-6 relative, combine within the combine tolerance.

The shapes vary everything the interface allows: ranks, experts per rank,
R up to min(E, 32), tokens per rank (including counts that are not multiples
of 32), row widths, row and output dtypes, score function, bias,
renormalisation, and capacities small enough to overflow."""
import random

import pytest

import oracle
from combine_moe_route_topk_gb300 import workloads as W
import sweep_params as S
from test_parity_gpu import _compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()


def _shapes(n, seed=20261202):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.choice([1, 2, 3, 4, 5, 8, 16])
        L = rng.choice([1, 2, 3, 4, 8, 16, 64])
        E = min(N * L, 1024 // N * N)
        R = rng.randint(1, min(E, 32))
        T = rng.choice([1, 7, 32, 33, 100, 257])
        x_dtype = rng.choice([W.BF16, W.BF16, W.F32, W.FP8E4M3_BLK128])
        if x_dtype == W.FP8E4M3_BLK128:
            H = 128 * rng.randint(1, 3)
            y_dtype, op = W.BF16, W.EXPERT_DEQUANT
        else:
            H = 8 * rng.randint(1, 64)
            y_dtype = rng.choice([x_dtype, W.F32 if x_dtype == W.BF16 else W.BF16])
            op = rng.choice([W.EXPERT_IDENTITY, W.EXPERT_SCALE])
        bound = N * T * max(R, E // N)
        cap = 0 if rng.random() < 0.75 else max(1, bound // rng.choice([8, 32, 64]))
        out.append(W.Workload(f"rand{i}", N=N, T=T, E=E, R=R, H=H, x_dtype=x_dtype,
                              y_dtype=y_dtype, expert_op=op,
                              score_fn=rng.choice([W.SOFTMAX, W.SIGMOID]),
                              renormalize=rng.random() < 0.5,
                              bias=rng.choice(["none", "normal"]), cap_rows=cap, seed=1000 + i))
    return out


def _large_shapes(n, seed=77):
    """Batches of several thousand tokens (the count kernel's 1024-thread
    blocks and several tiles of tokens per block), narrow rows."""
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.choice([1, 2, 3, 4, 8])
        E = N * rng.choice([1, 3, 5, 16, 32])
        R = rng.randint(1, min(E, 32))
        T = rng.randint(4097 // N + 1, 40000 // N)
        out.append(W.Workload(f"large{i}", N=N, T=T, E=E, R=R, H=8 * rng.randint(1, 8),
                              score_fn=rng.choice([W.SOFTMAX, W.SIGMOID]),
                              renormalize=rng.random() < 0.5, bias=rng.choice(["none", "normal"]),
                              seed=6000 + i))
    return out


SHAPES = _shapes(S.count(24), S.seed(20261202)) + _large_shapes(S.count(6), S.seed(77))


@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
def test_random_shape(w):
    gr, _, _ = _compare(w, W.make_inputs(w))
    assert gr.status in (oracle.OK, oracle.ERR_CAPACITY)
