"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test fixes the oracle to a fact the pages or mathematics give:
hand-worked golden cases (tests/golden/), closed forms, invariants, special
cases that reduce to a library routine, and brute force on tiny inputs by a
different algorithm (a global sort instead of running counters).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_topk_gb300 import workloads as W

from conftest import GOLDEN

SCORE = {"softmax": oracle.SOFTMAX, "sigmoid": oracle.SIGMOID,
         "softmax_bias_select": oracle.SOFTMAX | oracle.BIAS_SELECT_ONLY,
         "sigmoid_bias_select": oracle.SIGMOID | oracle.BIAS_SELECT_ONLY}


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)["cases"]


# --------------------------------------------------------------------------
# route top-k
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden("route_cases.json"), ids=lambda c: c["name"])
def test_route_golden(case):
    logits = np.array(case["logits"], np.float32)
    bias = None if case["bias"] is None else np.array(case["bias"], np.float32)
    idx, w, _ = oracle.route(logits, bias, case["R"], SCORE[case["score_fn"]],
                             case["renormalize"])
    assert idx.tolist() == case["topk_idx"]
    np.testing.assert_allclose(w, np.array(case["topk_w"]), rtol=case["tol"], atol=0)


def _lexsort_topk(z, R):
    # numpy's stable lexsort on (index, -z): a library routine independent of
    # the oracle's comparator sort
    out = np.empty((z.shape[0], R), np.int64)
    e = np.arange(z.shape[1])
    for g in range(z.shape[0]):
        out[g] = np.lexsort((e, -z[g].astype(np.float64)))[:R]
    return out


@pytest.mark.parametrize("E,R,tie_every,with_bias", [(16, 2, 3, False), (37, 5, 2, True),
                                                     (256, 8, 4, True), (8, 8, 1, False)])
def test_route_selection_matches_lexsort(E, R, tie_every, with_bias):
    w = W.Workload("t", N=1, T=97, E=E, R=R, H=8, bias="normal" if with_bias else "none",
                   seed=E)
    inp = W.make_inputs(w, tie_every=tie_every)
    logits = inp.logits.numpy()
    bias = None if inp.bias is None else inp.bias.numpy()
    z = logits + (bias if bias is not None else np.float32(0))  # float32 add
    assert z.dtype == np.float32
    idx, _, _ = oracle.route(logits, bias, R, oracle.SOFTMAX, False)
    np.testing.assert_array_equal(idx, _lexsort_topk(z, R))


def test_route_softmax_sums_to_one_over_all_experts():
    # with R = E and no renormalisation the weights are the full softmax
    w = W.Workload("t", N=1, T=64, E=24, R=24, H=8, seed=3)
    inp = W.make_inputs(w)
    _, wt, w64 = oracle.route(inp.logits.numpy(), None, 24, oracle.SOFTMAX, False)
    np.testing.assert_allclose(w64.sum(1), 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(wt.astype(np.float64).sum(1), 1.0, rtol=0, atol=24 * 6e-8)


def test_route_softmax_ratio_closed_form():
    # p_a / p_b = exp(z_a - z_b) for any two experts (shift invariance)
    w = W.Workload("t", N=1, T=32, E=40, R=6, H=8, bias="normal", seed=5)
    inp = W.make_inputs(w)
    logits, bias = inp.logits.numpy(), inp.bias.numpy()
    z = (logits + bias).astype(np.float64)
    idx, _, w64 = oracle.route(logits, bias, 6, oracle.SOFTMAX, False)
    for g in range(32):
        for k in range(1, 6):
            want = math.exp(z[g, idx[g, k]] - z[g, idx[g, 0]])
            assert w64[g, k] / w64[g, 0] == pytest.approx(want, rel=1e-12)
        # and the top weight against the full denominator
        den = np.exp(z[g] - z[g].max()).sum()
        assert w64[g, 0] == pytest.approx(1.0 / den, rel=1e-12)


@pytest.mark.parametrize("fn", [oracle.SOFTMAX, oracle.SIGMOID])
def test_route_bias_select_without_bias_is_the_default_reading(fn):
    # scores are monotone in the logit, so with no bias the flag changes
    # neither the selection nor (no bias to add) the weights
    w = W.Workload("t", N=1, T=80, E=48, R=6, H=8, seed=11)
    logits = W.make_inputs(w).logits.numpy()
    a = oracle.route(logits, None, 6, fn, True)
    b = oracle.route(logits, None, 6, fn | oracle.BIAS_SELECT_ONLY, True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_allclose(a[2], b[2], rtol=1e-12, atol=0)


def test_route_bias_select_weights_are_raw_scores():
    # a bias of +100 forces a chosen set of experts into the selection; their
    # weights stay the sigmoid / softmax of the raw logits (scipy's expit and
    # softmax), which adding the bias to the logit would not give
    special = pytest.importorskip("scipy.special")
    w = W.Workload("t", N=1, T=50, E=32, R=4, H=8, seed=12)
    logits = W.make_inputs(w).logits.numpy()
    forced = [3, 17, 18, 30]
    bias = np.zeros(32, np.float32)
    bias[forced] = 100.0
    for fn, ref in [(oracle.SIGMOID, special.expit(logits.astype(np.float64))),
                    (oracle.SOFTMAX, special.softmax(logits.astype(np.float64), axis=1))]:
        idx, _, w64 = oracle.route(logits, bias, 4, fn | oracle.BIAS_SELECT_ONLY, False)
        assert all(sorted(r) == forced for r in idx.tolist())
        np.testing.assert_allclose(w64, np.take_along_axis(ref, idx.astype(np.int64), 1),
                                   rtol=1e-12, atol=0)
        # and the selection order follows the float keys (float score + bias)
        keys = ref.astype(np.float32) + bias
        assert keys.dtype == np.float32
        np.testing.assert_array_equal(idx, _lexsort_topk(keys, 4))


def test_route_sigmoid_symmetry_and_monotone():
    # sigmoid(z) + sigmoid(-z) = 1; weights fall along the selection order
    logits = np.array([[0.3, -0.3, 2.0, -2.0, 0.0, 5.0, -5.0, 1.0]], np.float32)
    idx, _, w64 = oracle.route(logits, None, 8, oracle.SIGMOID, False)
    by_e = {int(e): w64[0, k] for k, e in enumerate(idx[0])}
    for a, b in [(0, 1), (2, 3), (5, 6)]:
        assert by_e[a] + by_e[b] == pytest.approx(1.0, abs=1e-15)
    assert by_e[4] == 0.5
    assert np.all(np.diff(w64[0]) <= 0)


@pytest.mark.parametrize("score", [oracle.SOFTMAX, oracle.SIGMOID])
def test_route_renorm_is_proportional_and_sums_to_one(score):
    w = W.Workload("t", N=1, T=50, E=64, R=8, H=8, seed=11)
    inp = W.make_inputs(w)
    _, _, raw = oracle.route(inp.logits.numpy(), None, 8, score, False)
    _, wt, ren = oracle.route(inp.logits.numpy(), None, 8, score, True)
    np.testing.assert_allclose(ren.sum(1), 1.0, atol=1e-12)
    np.testing.assert_allclose(ren, raw / raw.sum(1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(wt, ren, rtol=6e-8)


# --------------------------------------------------------------------------
# number formats used by the harness expert op
# --------------------------------------------------------------------------

def test_fp8_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.fp8e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(0)
    v = torch.cat([torch.randn(20000, generator=g) * 10 ** torch.randint(-5, 6, (20000,), generator=g),
                   torch.tensor([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65504.0, 1e-40,
                                 3.4e38, -3.4e38])])
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16_bits(float(t)) for t in v.tolist()], np.uint16)
    np.testing.assert_array_equal(got, ref)


# --------------------------------------------------------------------------
# dispatch count
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden("count_cases.json"), ids=lambda c: c["name"])
def test_count_golden(case):
    out, st = oracle.count(case["N"], case["T"], case["E"], case["cap"],
                           np.array(case["topk_idx"], np.int32))
    assert st == case["status"]
    for k in ("expert_counts", "expert_offsets", "rank_counts", "rank_offsets",
              "send_counts", "pos"):
        assert out[k].tolist() == case[k], k


def _bruteforce_count(N, T, E, cap, idx):
    """Independent restatement: list every valid pair, sort the list by
    (rank, expert, token, k) and hand out rows in that order."""
    NT, R = idx.shape
    L = E // N
    pairs = []
    for g in range(NT):
        seen = set()
        for k in range(R):
            e = int(idx[g, k])
            if 0 <= e < E and e not in seen:
                pairs.append((e // L, e, g, k))
            seen.add(e)
    pairs.sort()
    pos = -np.ones((NT, R), np.int64)
    used = [0] * N
    for (d, e, g, k) in pairs:
        if used[d] < cap:
            pos[g, k] = d * cap + used[d]
        used[d] += 1
    counts = np.bincount([p[1] for p in pairs], minlength=E)
    send = np.zeros((N, N), np.int64)
    for (d, e, g, k) in pairs:
        send[g // T, d] += 1
    return pos, counts, send


@pytest.mark.parametrize("N,T,E,R,cap", [(4, 9, 16, 2, 0), (3, 17, 12, 4, 0), (2, 33, 8, 8, 0),
                                         (4, 16, 16, 3, 10), (1, 40, 32, 5, 0)])
def test_count_matches_bruteforce(N, T, E, R, cap):
    rng = np.random.default_rng(N * 100 + T)
    NT = N * T
    idx = np.stack([rng.permutation(E)[:R] for _ in range(NT)]).astype(np.int32)
    cap = cap or N * T * max(R, E // N)
    out, st = oracle.count(N, T, E, cap, idx)
    pos, counts, send = _bruteforce_count(N, T, E, cap, idx)
    np.testing.assert_array_equal(out["pos"], pos)
    np.testing.assert_array_equal(out["expert_counts"], counts)
    np.testing.assert_array_equal(out["send_counts"], send)
    np.testing.assert_array_equal(out["expert_offsets"], np.concatenate([[0], np.cumsum(counts)]))
    rc = counts.reshape(N, E // N).sum(1)
    np.testing.assert_array_equal(out["rank_counts"], rc)
    np.testing.assert_array_equal(out["rank_offsets"], np.concatenate([[0], np.cumsum(rc)]))
    assert st == (oracle.ERR_CAPACITY if rc.max() > cap else oracle.OK)


def check_count_invariants(w, idx, out, cap):
    """Invariants every correct dispatch count satisfies (also used on GPU output)."""
    N, T, E, R = w.N, w.T, w.E, w.R
    L = E // N
    NT = N * T
    counts = out["expert_counts"].astype(np.int64)
    assert counts.sum() == NT * R                                   # every pair counted
    assert out["expert_offsets"][0] == 0
    np.testing.assert_array_equal(np.diff(out["expert_offsets"]), counts)  # exclusive scan
    rc = out["rank_counts"].astype(np.int64)
    np.testing.assert_array_equal(rc, counts.reshape(N, L).sum(1))
    np.testing.assert_array_equal(np.diff(out["rank_offsets"]), rc)
    # receive bound of the pages, and the tighter min(R, E/N) form
    assert rc.max() <= N * T * min(R, L) <= N * T * max(R, L)
    assert cap >= rc.max()
    sc = out["send_counts"].astype(np.int64)
    np.testing.assert_array_equal(sc.sum(1), np.full(N, T * R))
    np.testing.assert_array_equal(sc.sum(0), rc)
    pos = out["pos"].astype(np.int64)
    assert (pos >= 0).all()
    # bijection onto the occupied rows of each rank region
    d_of = idx // L
    assert (pos // cap == d_of).all()
    local = pos % cap
    flat = pos.ravel()
    assert np.unique(flat).size == flat.size
    for d in range(N):
        assert np.array_equal(np.sort(local[d_of == d]), np.arange(rc[d]))
    # each row within its expert's span, tokens ascending inside an expert
    base = out["expert_offsets"][idx] - out["rank_offsets"][d_of]
    assert (local >= base).all() and (local < base + counts[idx]).all()
    g_of = np.repeat(np.arange(NT), R).reshape(NT, R)
    order = np.argsort(flat, kind="stable")
    e_sorted = idx.ravel()[order]
    g_sorted = g_of.ravel()[order]
    same = e_sorted[1:] == e_sorted[:-1]
    assert (g_sorted[1:][same] > g_sorted[:-1][same]).all()


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_count_invariants_full_size(name):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w.replace(H=8, x_dtype=W.F32))   # routing only: skip the big x
    bias = None if inp.bias is None else inp.bias.numpy()
    idx, _, _ = oracle.route(inp.logits.numpy(), bias, w.R, w.score_fn, w.renormalize)
    cap = W.default_cap(w)
    out, st = oracle.count(w.N, w.T, w.E, cap, idx)
    assert st == oracle.OK
    check_count_invariants(w, idx, out, cap)
    # mean tokens per expert N*T*R/E (the pages' m formula)
    assert out["expert_counts"].mean() == w.NT * w.R / w.E


def test_skewed_bias_gives_about_half_to_top_five_percent():
    w = W.WORKLOADS["skewed"]
    inp = W.make_inputs(w.replace(H=8, x_dtype=W.F32))
    idx, _, _ = oracle.route(inp.logits.numpy(), inp.bias.numpy(), w.R, w.score_fn,
                             w.renormalize)
    c = np.bincount(idx.ravel(), minlength=w.E)
    share = W.log_zipf_top_share(torch.from_numpy(c))
    assert 0.47 <= share <= 0.53, share


# --------------------------------------------------------------------------
# pack
# --------------------------------------------------------------------------

@pytest.mark.parametrize("x_dtype", [W.BF16, W.F32, W.FP8E4M3_BLK128])
def test_pack_rows_are_copies_of_their_source(x_dtype):
    w = W.Workload("t", N=4, T=23, E=16, R=3, H=256, x_dtype=x_dtype, seed=2)
    inp = W.make_inputs(w)
    idx, _, _ = oracle.route(inp.logits.numpy(), None, w.R, 0, False)
    cap = W.default_cap(w)
    out, _ = oracle.count(w.N, w.T, w.E, cap, idx)
    xb = oracle.x_as_bytes(inp.x)
    xs = None if inp.x_scales is None else inp.x_scales.numpy()
    px, ps, src = oracle.pack(xb, xs, out["pos"], out["rank_offsets"], cap)
    assert (src >= 0).all() and np.unique(src).size == src.size == w.NT * w.R
    g, k = src // w.R, src % w.R
    np.testing.assert_array_equal(px, xb[g])
    if xs is not None:
        np.testing.assert_array_equal(ps, xs[g])
    # the compact row of pos[g][k] is exactly where src says (g, k) went
    d, local = out["pos"][g, k] // cap, out["pos"][g, k] % cap
    np.testing.assert_array_equal(out["rank_offsets"][d] + local, np.arange(src.size))


# --------------------------------------------------------------------------
# combine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden("combine_cases.json"), ids=lambda c: c["name"])
def test_combine_golden(case):
    idx = np.array(case["topk_idx"], np.int32)
    tw = np.array(case["topk_w"], np.float32)
    x = torch.tensor(case["x"], dtype=torch.float32)
    cnt, st = oracle.count(case["N"], case["T"], case["E"], case["cap"], idx)
    assert st == oracle.OK
    px, ps, src = oracle.pack(oracle.x_as_bytes(x), None, cnt["pos"], cnt["rank_offsets"],
                              case["cap"])
    y = oracle.expert_op(case["expert_op"], px, ps, src, idx, case["H"], oracle.F32, oracle.F32)
    out, _ = oracle.combine(y, oracle.F32, cnt["pos"], cnt["rank_offsets"], tw, case["cap"],
                            case["H"])
    np.testing.assert_array_equal(out, np.array(case["out"]))


def _path(w, inp):
    return oracle.run(w, inp)


@pytest.mark.parametrize("x_dtype", [W.BF16, W.F32])
def test_combine_identity_closed_form(x_dtype):
    # identity expert: out[g] = x[g] * sum_k w[g][k]
    w = W.Workload("t", N=4, T=31, E=32, R=4, H=64, x_dtype=x_dtype, y_dtype=x_dtype, seed=7)
    inp = W.make_inputs(w)
    r = _path(w, inp)
    xd = inp.x.to(torch.float64).numpy()
    want = xd * r["topk_w"].astype(np.float64).sum(1, keepdims=True)
    np.testing.assert_allclose(r["out"], want, rtol=1e-14, atol=1e-300)


def test_combine_renormalised_identity_returns_x():
    w = W.Workload("t", N=2, T=40, E=16, R=4, H=32, renormalize=True, seed=9)
    inp = W.make_inputs(w)
    r = _path(w, inp)
    np.testing.assert_allclose(r["out"], inp.x.to(torch.float64).numpy(), rtol=4 * 2 ** -24)


def test_combine_scale_closed_form():
    # scale expert: out[g] = x[g] * sum_k w_k s_{e_k} (bf16-exact scales, f32 rows)
    w = W.Workload("t", N=4, T=19, E=28, R=5, H=48, x_dtype=W.F32, y_dtype=W.F32,
                   expert_op=W.EXPERT_SCALE, seed=13)
    inp = W.make_inputs(w)
    r = _path(w, inp)
    s = np.array([W.expert_scale_value(e) for e in range(w.E)])
    xd = inp.x.to(torch.float64).numpy()
    # y = fl32(x * s) is exact here only up to float rounding: compare with 1 ulp
    factor = (r["topk_w"].astype(np.float64) * s[r["topk_idx"]]).sum(1, keepdims=True)
    np.testing.assert_allclose(r["out"], xd * factor, rtol=2 ** -23)


def test_combine_single_expert_unit_weight_is_a_gather():
    # R = 1 with weight 1 is a pure permutation inverse: out == x bit for bit
    w = W.Workload("t", N=4, T=25, E=8, R=1, H=40, x_dtype=W.F32, y_dtype=W.F32, seed=17)
    inp = W.make_inputs(w)
    idx, _, _ = oracle.route(inp.logits.numpy(), None, 1, 0, False)
    cap = W.default_cap(w)
    cnt, _ = oracle.count(w.N, w.T, w.E, cap, idx)
    px, ps, src = oracle.pack(oracle.x_as_bytes(inp.x), None, cnt["pos"], cnt["rank_offsets"], cap)
    y = oracle.expert_op("identity", px, ps, src, idx, w.H, oracle.F32, oracle.F32)
    out, _ = oracle.combine(y, oracle.F32, cnt["pos"], cnt["rank_offsets"],
                            np.ones((w.NT, 1), np.float32), cap, w.H)
    np.testing.assert_array_equal(out, inp.x.to(torch.float64).numpy())


def test_dequant_expert_matches_library_decode():
    # fp8 dequant expert: bf16(fl32(decode(q) * scale)) against torch's decode
    w = W.Workload("t", N=2, T=8, E=8, R=2, H=256, x_dtype=W.FP8E4M3_BLK128,
                   expert_op=W.EXPERT_DEQUANT, seed=21)
    inp = W.make_inputs(w)
    r = _path(w, inp)
    g = r["packed_src"] // w.R
    q = inp.x.view(torch.float8_e4m3fn)[torch.from_numpy(g)].to(torch.float32)
    sc = inp.x_scales[torch.from_numpy(g)].repeat_interleave(128, dim=1)
    want = (q * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(r["y"], want)


# --------------------------------------------------------------------------
# fp8 block quantisation (fused into the quantising pack)
# --------------------------------------------------------------------------

def _e4m3_magnitudes():
    return np.array([oracle.fp8e4m3_decode(c) for c in range(127)])


def test_e4m3_encode_is_nearest_code_ties_to_even():
    mags = _e4m3_magnitudes()
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.normal(0, 50, 3000), rng.normal(0, 0.01, 2000),
                           (mags[1:] + mags[:-1]) / 2,            # exact midpoints
                           -(mags[1:] + mags[:-1]) / 2, mags, -mags,
                           [0.0, -0.0, 447.9, 448.0, 460.0, 470.0, 1e6, -1e6]]).astype(np.float32)
    for v in vals.tolist():
        c = oracle.f32_to_fp8e4m3(v)
        a = abs(v)
        if a > 448:
            assert c & 0x7F == 126
        else:
            d = np.abs(mags - a)
            best = np.flatnonzero(d == d.min())
            want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
            assert c & 0x7F == want, (v, c, want)
        assert (c >> 7) == (1 if np.signbit(np.float32(v)) else 0)


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(5)
    v = torch.cat([torch.randn(20000, generator=g) * 30, torch.randn(5000, generator=g) * 1e-2])
    v = v.clamp(-448, 448)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_fp8e4m3(float(t)) for t in v.tolist()], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_block_quantisation_properties():
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(6, 512, generator=g) * torch.tensor([1.0, 1e-3, 30.0, 0.0]).repeat_interleave(128)).to(torch.bfloat16)
    codes, scales = oracle.quantize_rows(x)
    xf = x.to(torch.float64).numpy().reshape(6, 4, 128)
    amax = np.abs(xf).max(axis=2)
    np.testing.assert_array_equal(scales, (amax.astype(np.float32) / np.float32(448)))
    dec = np.vectorize(oracle.fp8e4m3_decode)(codes).reshape(6, 4, 128)
    for r in range(6):
        for blk in range(4):
            if amax[r, blk] == 0:
                assert (codes.reshape(6, 4, 128)[r, blk] == 0).all() and scales[r, blk] == 0
                continue
            # the largest element lands on +-448; the rest within half a code step
            assert np.abs(dec[r, blk]).max() == 448.0
            err = np.abs(dec[r, blk] * scales[r, blk] - xf[r, blk])
            assert (err <= np.abs(xf[r, blk]) * 2.0 ** -4 + scales[r, blk] * 2.0 ** -10 + 1e-30).all()


# --------------------------------------------------------------------------
# accumulation per destination rank (send-side partials, EP-only local part)
# --------------------------------------------------------------------------

def _routed(w):
    inp = W.make_inputs(w)
    r = oracle.run(w, inp)
    return inp, r


def test_rank_accumulations_sum_to_the_combine():
    # sum over ranks of the local accumulations = the combine (closed form)
    w = W.Workload("t", N=4, T=21, E=16, R=5, H=40, x_dtype=W.F32, y_dtype=W.F32,
                   expert_op=W.EXPERT_SCALE, seed=23)
    inp, r = _routed(w)
    tot = sum(oracle.combine_rank(r["y"], w.y_dtype, r["pos"], r["rank_offsets"], r["topk_w"],
                                  r["cap"], w.H, d) for d in range(w.N))
    np.testing.assert_allclose(tot, r["out"], rtol=1e-13, atol=1e-300)


def test_rank_accumulation_only_sees_local_pairs():
    # identity expert: out_d[g] = x[g] * (sum of the weights of g's pairs on d)
    w = W.Workload("t", N=4, T=17, E=16, R=3, H=24, x_dtype=W.F32, y_dtype=W.F32, seed=29)
    inp, r = _routed(w)
    L = w.E // w.N
    xd = inp.x.to(torch.float64).numpy()
    for d in range(w.N):
        got = oracle.combine_rank(r["y"], w.y_dtype, r["pos"], r["rank_offsets"], r["topk_w"],
                                  r["cap"], w.H, d)
        wsum = (r["topk_w"].astype(np.float64) * (r["topk_idx"] // L == d)).sum(1, keepdims=True)
        np.testing.assert_allclose(got, xd * wsum, rtol=1e-14, atol=1e-300)


def test_partials_slots_follow_first_appearance_and_sum_to_combine():
    w = W.Workload("t", N=4, T=19, E=32, R=6, H=32, x_dtype=W.F32, y_dtype=W.F32, seed=37)
    inp, r = _routed(w)
    part, slot = oracle.combine_partials(r["y"], w.y_dtype, r["pos"], r["rank_offsets"],
                                         r["topk_w"], r["cap"], w.H, w.N)
    L = w.E // w.N
    for g in range(w.NT):
        ranks = []
        for k in range(w.R):
            d = int(r["topk_idx"][g, k]) // L
            if d not in ranks:
                ranks.append(d)
        assert slot[g].tolist() == ranks + [-1] * (min(w.R, w.N) - len(ranks))
    out = oracle.reduce_partials(part, slot, w.y_dtype)
    # f32 partials: each rounded once to float
    np.testing.assert_allclose(out, r["out"], rtol=3 * 2.0 ** -24 * w.R, atol=1e-30)


def test_bf16_partials_round_each_rank_sum_once():
    w = W.Workload("t", N=2, T=16, E=8, R=4, H=16, seed=41)
    inp, r = _routed(w)
    part, slot = oracle.combine_partials(r["y"], w.y_dtype, r["pos"], r["rank_offsets"],
                                         r["topk_w"], r["cap"], w.H, w.N)
    for j in range(part.shape[1]):
        for g in range(w.NT):
            d = slot[g, j]
            if d < 0:
                assert (part[g, j] == 0).all()
                continue
            want = oracle.combine_rank(r["y"], w.y_dtype, r["pos"][g:g + 1], r["rank_offsets"],
                                       r["topk_w"][g:g + 1], r["cap"], w.H, int(d))[0]
            bits = np.array([oracle.f32_to_bf16_bits(float(np.float32(v))) for v in want], np.uint16)
            np.testing.assert_array_equal(part[g, j], bits)
