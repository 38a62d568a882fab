"""Host-side checks of the C ABI: the library builds for sm_103a, loads,
exports every entry point the header declares, sizes buffers, and rejects bad
arguments before touching the GPU.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

import combine_moe_route_topk_gb300 as moe
from combine_moe_route_topk_gb300 import _build
from combine_moe_route_topk_gb300 import workloads as W

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe_route.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("moe_buffer_sizes", "moe_route_topk", "moe_dispatch_count", "moe_dispatch_pack",
              "moe_combine", "moe_read_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_is_built_for_sm_103a_only():
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version(lib):
    # the library reports the version its header defines
    header = open(os.path.join(ROOT, "include", "moe_route.h")).read()
    assert f"#define MOE_VERSION {lib.moe_version()}" in header


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_buffer_sizes_follow_the_bound(lib, name):
    w = W.WORKLOADS[name]
    s = moe.buffer_sizes(moe.dims_of(w))
    L = w.E // w.N
    bound = w.N * w.T * max(w.R, L)
    assert s["bound_rows"] == bound == s["cap_rows"]
    assert s["total_pairs"] == w.NT * w.R
    rb = W.row_bytes(w)
    assert s["packed_x_bytes"] == w.N * bound * rb
    assert s["x_bytes"] == w.NT * rb
    assert s["pos_bytes"] == w.NT * w.R * 4
    assert s["send_counts_bytes"] == w.N * w.N * 4
    if w.x_dtype == W.FP8E4M3_BLK128:
        assert s["packed_scales_bytes"] == w.N * bound * (w.H // 128) * 4
    else:
        assert s["packed_scales_bytes"] == 0


def test_explicit_capacity_is_used(lib):
    s = moe.buffer_sizes(moe.make_dims(4, 64, 16, 2, 1024, cap_rows=100))
    assert s["cap_rows"] == 100 and s["bound_rows"] == 4 * 64 * 4


BAD_DIMS = [
    (dict(N=3, T=8, E=16, R=2, H=64), moe.MOE_ERR_INVALID_ARG, "multiple of N"),
    (dict(N=4, T=8, E=16, R=17, H=64), moe.MOE_ERR_INVALID_ARG, "exceeds E"),
    (dict(N=4, T=8, E=64, R=33, H=64), moe.MOE_ERR_UNSUPPORTED, "R<=32"),
    (dict(N=4, T=8, E=2048, R=2, H=64), moe.MOE_ERR_UNSUPPORTED, "E<=1024"),
    (dict(N=4, T=8, E=16, R=2, H=60), moe.MOE_ERR_INVALID_ARG, "multiple of 8"),
    (dict(N=4, T=8, E=16, R=2, H=64, x_dtype=moe.MOE_FP8E4M3_BLK128), moe.MOE_ERR_INVALID_ARG,
     "128"),
    (dict(N=4, T=8, E=16, R=2, H=64, x_dtype=7), moe.MOE_ERR_INVALID_ARG, "x_dtype"),
    (dict(N=4, T=8, E=16, R=2, H=64, y_dtype=moe.MOE_FP8E4M3_BLK128), moe.MOE_ERR_INVALID_ARG,
     "y_dtype"),
    (dict(N=0, T=8, E=16, R=2, H=64), moe.MOE_ERR_INVALID_ARG, "N>=1"),
    (dict(N=4, T=-1, E=16, R=2, H=64), moe.MOE_ERR_INVALID_ARG, "T>=0"),
    (dict(N=4, T=8, E=16, R=2, H=64, cap_rows=-5), moe.MOE_ERR_INVALID_ARG, "cap_rows"),
    (dict(N=64, T=100000, E=384, R=8, H=64), moe.MOE_ERR_UNSUPPORTED, "2^31"),
]


@pytest.mark.parametrize("kw,code,msg", BAD_DIMS)
def test_bad_dims_are_rejected_on_the_host(lib, kw, code, msg):
    d = moe.make_dims(**kw)
    s = moe.MoeSizes()
    assert lib.moe_buffer_sizes(ctypes.byref(d), ctypes.byref(s)) == code
    assert msg in lib.moe_last_error().decode()
    # every compute entry point validates the same way before any CUDA call
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert lib.moe_route_topk(ctypes.byref(d), fake, None, 0, 0, fake, fake, None) == code
    assert lib.moe_dispatch_count(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, fake,
                                  None) == code
    assert lib.moe_dispatch_pack(ctypes.byref(d), fake, fake, fake, fake, fake, fake, None) == code
    assert lib.moe_combine(ctypes.byref(d), fake, fake, fake, fake, None) == code


def test_quant_pack_rejects_non_bf16_rows_and_bad_h(lib):
    P = ctypes.c_void_p
    ok = P(0x10000)
    d = moe.make_dims(4, 8, 16, 2, 128, x_dtype=moe.MOE_F32)
    assert lib.moe_dispatch_pack_quant(ctypes.byref(d), ok, ok, ok, ok, ok, None) == moe.MOE_ERR_INVALID_ARG
    assert "MOE_BF16" in lib.moe_last_error().decode()
    d = moe.make_dims(4, 8, 16, 2, 64)
    assert lib.moe_dispatch_pack_quant(ctypes.byref(d), ok, ok, ok, ok, ok, None) == moe.MOE_ERR_INVALID_ARG
    assert "128" in lib.moe_last_error().decode()


def test_fused_dispatch_rejects_non_decode_shapes(lib):
    P = ctypes.c_void_p
    ok = P(0x10000)
    args = [ok] * 16
    # beyond the single-cluster path (N*T <= 512, E <= 256) the two-kernel
    # form's limits apply (R <= 32 is the interface's own limit)
    for kw, why in [(dict(N=4, T=4096, E=128, R=8, H=128), "4096"),
                    (dict(N=4, T=64, E=1024, R=8, H=128), "E > 512")]:
        d = moe.make_dims(**kw)
        assert lib.moe_dispatch_fused(ctypes.byref(d), ok, None, 0, 0, ok, None, *args[:11], None,
                                      ok, ok, None) == moe.MOE_ERR_UNSUPPORTED
        assert why in lib.moe_last_error().decode()


def test_fused_dispatch_accepts_empty_batches_of_any_shape(lib):
    # the shape check passes (an empty batch only runs the count step); with
    # no GPU the call then fails, if at all, only at the CUDA level
    P = ctypes.c_void_p
    ok = P(0x10000)
    args = [ok] * 16
    d = moe.make_dims(N=4, T=0, E=64, R=16, H=128)
    rc = lib.moe_dispatch_fused(ctypes.byref(d), None, None, 0, 0, None, None, *args[:11], None,
                                ok, ok, None)
    assert rc != moe.MOE_ERR_INVALID_ARG
    assert "use the separate calls" not in lib.moe_last_error().decode()


def test_fused_dispatch_takes_a_null_workspace_only_for_an_empty_batch(lib):
    P = ctypes.c_void_p
    ok = P(0x10000)

    def call(d):
        # logits, bias, score_fn, renormalize, x, x_scales, then topk_idx ..
        # packed_x (10 pointers), packed_scales (NULL: bf16 rows), packed_src,
        # a NULL workspace and the default stream
        ptrs = [ok] * 10 + [None, ok]
        return lib.moe_dispatch_fused(ctypes.byref(d), ok, None, 0, 0, ok, None, *ptrs, None, None)

    assert call(moe.make_dims(N=4, T=64, E=64, R=8, H=128)) == moe.MOE_ERR_INVALID_ARG
    assert "NULL" in lib.moe_last_error().decode()
    rc = call(moe.make_dims(N=4, T=0, E=64, R=8, H=128))
    assert rc != moe.MOE_ERR_INVALID_ARG  # no GPU here: at most a CUDA-level failure


def test_rows_wider_than_2_24_elements_are_unsupported(lib):
    d = moe.make_dims(2, 8, 4, 2, (1 << 24) + 8)
    s = moe.MoeSizes()
    assert lib.moe_buffer_sizes(ctypes.byref(d), ctypes.byref(s)) == moe.MOE_ERR_UNSUPPORTED
    assert "2^24" in lib.moe_last_error().decode()


def test_reserved_field_must_be_zero(lib):
    d = moe.make_dims(4, 8, 16, 2, 64)
    d.reserved = 1
    s = moe.MoeSizes()
    assert lib.moe_buffer_sizes(ctypes.byref(d), ctypes.byref(s)) == moe.MOE_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_are_rejected(lib):
    d = moe.make_dims(4, 8, 16, 2, 64)
    P = ctypes.c_void_p
    ok, odd, mis16 = P(0x10000), P(0x10002), P(0x10008)
    E_INV = moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk(ctypes.byref(d), None, None, 0, 0, ok, ok, None) == E_INV
    assert lib.moe_route_topk(ctypes.byref(d), odd, None, 0, 0, ok, ok, None) == E_INV
    assert lib.moe_route_topk(ctypes.byref(d), ok, None, 5, 0, ok, ok, None) == E_INV
    assert "score_fn" in lib.moe_last_error().decode()
    for bad in (0x20, 0x12, moe.MOE_BIAS_SELECT_ONLY | 2, -1):
        assert lib.moe_route_topk(ctypes.byref(d), ok, None, bad, 0, ok, ok, None) == E_INV
    assert lib.moe_dispatch_count(ctypes.byref(d), ok, ok, ok, ok, ok, ok, ok, None, None) == E_INV
    assert lib.moe_dispatch_pack(ctypes.byref(d), mis16, None, ok, ok, None, ok, None) == E_INV
    assert "16-byte" in lib.moe_last_error().decode()
    assert lib.moe_dispatch_pack(ctypes.byref(d), ok, None, ok, None, None, ok, None) == E_INV
    fp8 = moe.make_dims(4, 8, 16, 2, 128, x_dtype=moe.MOE_FP8E4M3_BLK128)
    assert lib.moe_dispatch_pack(ctypes.byref(fp8), ok, None, ok, ok, None, ok, None) == E_INV
    assert lib.moe_combine(ctypes.byref(d), ok, ok, ok, mis16, None) == E_INV
    assert lib.moe_read_status(None, None) == E_INV
    assert lib.moe_dispatch_pack(None, ok, None, ok, ok, None, ok, None) == E_INV


def test_binding_refuses_cpu_tensors(lib):
    import torch
    d = moe.make_dims(1, 4, 8, 2, 64)
    t = torch.zeros(4, 8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        moe.route_topk(d, t, None, 0, False, t, t)


def test_rank_entries_reject_ranks_outside_the_batch(lib):
    P = ctypes.c_void_p
    ok = P(0x10000)
    d = moe.make_dims(N=4, T=8, E=8, R=2, H=64)
    for rank in (-1, 4, 1 << 20):
        assert lib.moe_dispatch_pack_rank(ctypes.byref(d), rank, ok, None, ok, ok, None, ok,
                                          None) == moe.MOE_ERR_INVALID_ARG
        assert "outside [0, 4)" in lib.moe_last_error().decode()
        assert lib.moe_combine_rank(ctypes.byref(d), rank, ok, ok, ok, ok,
                                    None) == moe.MOE_ERR_INVALID_ARG
        assert "outside [0, 4)" in lib.moe_last_error().decode()


def _fused_workspace_layout(N, T, E):
    """The two-kernel fused dispatch's workspace, restated: a 256-byte header
    (the arrival counter), one byte per expert per route block, a u16 prefix
    per expert per chunk of 8 route blocks and, when source ranks are split
    over blocks (T > 32), a u16 send count per block and destination rank;
    every section padded to 256 bytes.  Route blocks hold at most 32 tokens
    and never cross a source rank."""
    a256 = lambda v: (v + 255) // 256 * 256
    Ep = (E + 15) // 16 * 16
    if T <= 32:
        B, split = -(-N // (32 // T)), False
    else:
        B, split = N * -(-T // 32), True
    return 256 + a256(B * Ep) + a256(-(-B // 8) * Ep * 2) + (a256(B * N * 2) if split else 0)


@pytest.mark.parametrize("N,T,E", [(32, 128, 256), (64, 64, 384), (16, 256, 512), (4, 160, 96), (512, 1, 512),
                                   (200, 5, 400), (48, 17, 96), (124, 33, 496), (8, 100, 64), (1, 32, 8)])
def test_fused_workspace_size(lib, N, T, E):
    s = moe.buffer_sizes(moe.make_dims(N, T, E, min(8, E), 64))
    assert s["fused_workspace_bytes"] == _fused_workspace_layout(N, T, E)


def test_fused_workspace_fits_the_static_scratch_and_is_zero_outside_the_fused_scope(lib):
    # the largest workspace of any batch the two-kernel form takes (N*T <=
    # 4096, E <= 512) is that of N = 124, T = 33, E = 496; the static array
    # of moe_dispatch_fused_static holds 256 KiB
    worst = 0
    for N in (1, 2, 4, 8, 16, 31, 62, 124, 128, 256, 512):
        for T in sorted({1, 2, 5, 16, 17, 31, 32, 33, 63, 64, 65, 100, 128, 4096 // N}):
            if T < 1 or N * T > 4096:
                continue
            E = 512 // N * N
            if E == 0:
                continue
            got = moe.buffer_sizes(moe.make_dims(N, T, E, min(8, E), 64))["fused_workspace_bytes"]
            assert got == _fused_workspace_layout(N, T, E), (N, T, E)
            worst = max(worst, got)
    assert worst <= 256 * 1024
    assert moe.buffer_sizes(moe.make_dims(124, 33, 496, 8, 64))["fused_workspace_bytes"] == 216064
    # no fused form with a workspace takes these: more than 4096 tokens, E > 512
    assert moe.buffer_sizes(moe.make_dims(4, 4096, 128, 8, 64))["fused_workspace_bytes"] == 0
    assert moe.buffer_sizes(moe.make_dims(4, 64, 1024, 8, 64))["fused_workspace_bytes"] == 0


@pytest.mark.parametrize("kw,code,msg", [
    (dict(N=4, T=64, E=64, R=8, H=128, x_dtype=moe.MOE_F32), moe.MOE_ERR_INVALID_ARG, "MOE_BF16"),
    (dict(N=4, T=64, E=64, R=8, H=136), moe.MOE_ERR_INVALID_ARG, "multiple of 128"),
    (dict(N=4, T=4096, E=64, R=8, H=128), moe.MOE_ERR_UNSUPPORTED, "4096"),
    (dict(N=4, T=64, E=1024, R=8, H=128), moe.MOE_ERR_UNSUPPORTED, "E > 512")])
def test_fused_quant_dispatch_rejects_bad_rows_and_non_decode_batches(lib, kw, code, msg):
    P = ctypes.c_void_p
    ok = P(0x10000)
    d = moe.make_dims(**kw)
    # logits, bias, score_fn, renormalize, x, then topk_idx .. packed_src
    # (12 pointers), the workspace and the stream
    assert lib.moe_dispatch_fused_quant(ctypes.byref(d), ok, None, 0, 0, ok, *([ok] * 12), ok, None) == code
    assert msg in lib.moe_last_error().decode()
