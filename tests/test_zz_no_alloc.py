"""The allocation-free fused dispatch, moe_dispatch_fused_static.

Some callers cannot allocate device memory at the moment they dispatch: a
plug-in running inside another framework's execution loop has no allocator
of its own, and serving code whose memory is fixed at start-up must not call
cudaMalloc on its hot path (it synchronises the device and can fail under
memory pressure).  For them moe_dispatch_fused_static runs the fused
route + count + pack with scratch that lives in the library itself.

The GPU test calls it through the C ABI twice in a row, on two different
batches, and checks every output of each call against moe_dispatch_fused
given a freshly allocated workspace.  The second call sees the scratch as
the first call left it, so anything that must start at zero and was not
cleared would show up there.  Integer outputs and packed rows must be equal
byte for byte; router weights within the relative 2e-6 that the other
parity tests allow (both calls run the same kernel, so they agree exactly
in practice).

This file sorts last so that a run stopping at its first failure has run
every other test before it.
"""
import dataclasses

import numpy as np
import pytest
import torch

import combine_moe_route_topk_gb300 as moe
from combine_moe_route_topk_gb300 import workloads as W
from gpu_path import TOPK_W_RTOL

OUTPUTS = ("topk_idx", "topk_w", "expert_counts", "expert_offsets", "rank_counts", "rank_offsets",
           "send_counts", "pos", "status", "packed_x", "packed_src")


def _dispatch(w: W.Workload, d: W.Inputs, static: bool) -> dict:
    dims = moe.dims_of(w)
    b = moe.Buffers(dims, device=d.logits.device)
    # every output starts from zero so that whole buffers can be compared
    for k in OUTPUTS:
        getattr(b, k).view(torch.uint8).zero_()
    args = (dims, d.logits, d.bias, w.score_fn, w.renormalize, d.x, d.x_scales, b.topk_idx,
            b.topk_w, b.expert_counts, b.expert_offsets, b.rank_counts, b.rank_offsets,
            b.send_counts, b.pos, b.status, b.packed_x, b.packed_scales, b.packed_src)
    if static:
        moe.dispatch_fused_static(*args)
    else:
        ws = torch.empty(b.sizes["fused_workspace_bytes"], dtype=torch.uint8, device=d.logits.device)
        moe.dispatch_fused(*args, ws)
    torch.cuda.synchronize()
    return {k: getattr(b, k).view(torch.uint8 if k == "packed_x" else getattr(b, k).dtype).cpu().numpy()
            for k in OUTPUTS}


@pytest.mark.gpu
def test_static_scratch_matches_allocated_workspace_on_two_calls_in_a_row():
    from combine_moe_route_topk_gb300 import _build
    _build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    base = W.WORKLOADS["dsv3_decode"]
    for seed in (base.seed + 101, base.seed + 202):
        w = dataclasses.replace(base, seed=seed)
        inp = W.make_inputs(w)
        d = W.Inputs(*(t.to(dev) if t is not None else None
                       for t in (inp.logits, inp.bias, inp.x, inp.x_scales)))
        got = _dispatch(w, d, static=True)
        want = _dispatch(w, d, static=False)
        assert int(want["status"][0]) == moe.MOE_OK
        for k in OUTPUTS:
            if k == "topk_w":
                np.testing.assert_allclose(got[k], want[k], rtol=TOPK_W_RTOL, atol=0, err_msg=k)
            else:
                np.testing.assert_array_equal(got[k], want[k], err_msg=f"{k} (seed {seed})")


def test_static_variant_rejects_shapes_the_fused_kernel_cannot_take():
    import ctypes
    lib = moe.lib()
    ok = ctypes.c_void_p(0x10000)
    d = moe.make_dims(N=4, T=64, E=1024, R=8, H=128)
    rc = lib.moe_dispatch_fused_static(ctypes.byref(d), ok, None, 0, 0, ok, None, *([ok] * 11),
                                       None, ok, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    assert "moe_dispatch_fused_static" in lib.moe_last_error().decode()
