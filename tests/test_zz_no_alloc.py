"""The allocation-free fused dispatch, moe_dispatch_fused_static.

Some callers cannot allocate device memory at the moment they dispatch: a
plug-in running inside another framework's execution loop has no allocator
of its own, and serving code whose memory is fixed at start-up must not call
cudaMalloc on its hot path (it synchronises the device and can fail under
memory pressure).  For them moe_dispatch_fused_static runs the fused
route + count + pack with scratch that lives in the library itself.

The GPU test calls it through the C ABI several times in a row, on batches
of different shapes, and then checks every output of each call against
moe_dispatch_fused given a freshly allocated, zero-filled workspace.
The calls shrink from the widest scratch use to a narrower one: 512
experts and 128 route blocks, then 256 experts and 128 blocks, then 96
experts, 4 ranks and 20 blocks.  Each later call sees the scratch as the
previous one left it, including histogram, prefix and send-count words past
its own experts, ranks and blocks, so a call that read anything it had not
written first, or that left the arrival counter off zero, would show up
there.  Integer outputs and packed rows must be equal
byte for byte; router weights within the relative 2e-6 that the other
parity tests allow (both calls run the same kernel, so they agree exactly
in practice).

This file sorts last so that a run stopping at its first failure has run
every other test before it.
"""
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
        ws = torch.zeros(b.sizes["fused_workspace_bytes"], dtype=torch.uint8, device=d.logits.device)
        moe.dispatch_fused(*args, ws)
    torch.cuda.synchronize()
    return {k: getattr(b, k).view(torch.uint8 if k == "packed_x" else getattr(b, k).dtype).cpu().numpy()
            for k in OUTPUTS}


# batches of the two-kernel form (more than 512 tokens), widest scratch use
# first.  Receive regions of 4096 rows per rank (the
# largest rank receives 2774, 1945 and 1001 rows) keep the buffers compared
# on the host small; the capacity does not change what the scratch holds.
STATIC_SEQUENCE = (
    W.Workload("e512", N=16, T=256, E=512, R=8, H=1024, score_fn=W.SIGMOID, bias="normal",
               renormalize=True, cap_rows=4096, seed=301),
    W.WORKLOADS["dsv3_decode"].replace(seed=302, cap_rows=4096),
    W.Workload("e96", N=4, T=160, E=96, R=6, H=2048, renormalize=True, cap_rows=4096, seed=303),
)


@pytest.mark.gpu
def test_static_scratch_matches_allocated_workspace_on_calls_in_a_row():
    from combine_moe_route_topk_gb300 import _build
    _build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    inputs = []
    for w in STATIC_SEQUENCE:
        inp = W.make_inputs(w)
        inputs.append(W.Inputs(*(t.to(dev) if t is not None else None
                                 for t in (inp.logits, inp.bias, inp.x, inp.x_scales))))
    # the static calls back to back, then the same batches with a workspace
    got = [_dispatch(w, d, static=True) for w, d in zip(STATIC_SEQUENCE, inputs)]
    for w, d, g in zip(STATIC_SEQUENCE, inputs, got):
        want = _dispatch(w, d, static=False)
        assert int(want["status"][0]) == moe.MOE_OK, w.name
        for k in OUTPUTS:
            if k == "topk_w":
                np.testing.assert_allclose(g[k], want[k], rtol=TOPK_W_RTOL, atol=0,
                                           err_msg=f"{k} ({w.name})")
            else:
                np.testing.assert_array_equal(g[k], want[k], err_msg=f"{k} ({w.name})")


def test_static_variant_rejects_shapes_the_fused_kernel_cannot_take():
    import ctypes
    lib = moe.lib()
    ok = ctypes.c_void_p(0x10000)
    d = moe.make_dims(N=4, T=64, E=1024, R=8, H=128)
    rc = lib.moe_dispatch_fused_static(ctypes.byref(d), ok, None, 0, 0, ok, None, *([ok] * 11),
                                       None, ok, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    assert "moe_dispatch_fused_static" in lib.moe_last_error().decode()
