"""The library keeps a few facts per CUDA context on the host: kernel
attributes that a launch needs (more than 48 KB of dynamic shared memory,
non-portable cluster sizes) and the device address of its scratch array.
cudaDeviceReset ends the context and the next call runs in a new one, where
those attributes are unset; the caches key on the context, so calls after a
reset set them again.  This runs in a child process that uses the C ABI and
the CUDA runtime through ctypes only (PyTorch's allocator does not survive a
device reset): the count of a 5120-token batch with E = 512 (1024-thread
blocks, about 96 KB of shared memory) and the fused dispatch of a 256-token
batch (single cluster) and a 1024-token batch (route kernel that counts,
then the pack kernel), before and after a reset, with identical outputs."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes, os, sys
import numpy as np
root = sys.argv[1]
lib = ctypes.CDLL(os.path.join(root, "combine_moe_route_topk_gb300", "libmoe_route.so"))
rt_path = next(l.split()[-1] for l in open("/proc/self/maps") if "libcudart.so" in l)
rt = ctypes.CDLL(rt_path)
P, i64 = ctypes.c_void_p, ctypes.c_int64

class Dims(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int32), ("T", ctypes.c_int32), ("E", ctypes.c_int32), ("R", ctypes.c_int32),
                ("H", ctypes.c_int32), ("x_dtype", ctypes.c_int32), ("y_dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("cap_rows", ctypes.c_int64)]

def dmalloc(nbytes):
    p = P()
    assert rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(max(nbytes, 16))) == 0
    return p

def h2d(p, a):
    assert rt.cudaMemcpy(p, a.ctypes.data_as(P), ctypes.c_size_t(a.nbytes), 1) == 0

def d2h(a, p):
    assert rt.cudaMemcpy(a.ctypes.data_as(P), p, ctypes.c_size_t(a.nbytes), 2) == 0

rng = np.random.default_rng(5)

def count_round():
    N, T, E, R = 4, 1280, 512, 8
    NT = N * T
    idx = np.stack([rng.permutation(E)[:R] for _ in range(NT)]).astype(np.int32)
    d = Dims(N, T, E, R, 64, 0, 0, 0, 0)
    bufs = {k: dmalloc(n) for k, n in dict(idx=idx.nbytes, ec=4 * E, eo=4 * (E + 1), rc=4 * N,
                                           ro=4 * (N + 1), sc=4 * N * N, pos=idx.nbytes, st=4).items()}
    h2d(bufs["idx"], idx)
    rc = lib.moe_dispatch_count(ctypes.byref(d), bufs["idx"], bufs["ec"], bufs["eo"], bufs["rc"], bufs["ro"],
                                bufs["sc"], bufs["pos"], bufs["st"], None)
    assert rc == 0, (rc, lib.moe_last_error())
    assert rt.cudaDeviceSynchronize() == 0
    pos = np.empty_like(idx)
    d2h(pos, bufs["pos"])
    ec = np.empty(E, np.int32)
    d2h(ec, bufs["ec"])
    for p in bufs.values():
        rt.cudaFree(p)
    return pos, ec

def fused_round(T):
    # T = 64: 256 tokens, the single-cluster kernel; T = 256: 1024 tokens,
    # the route kernel that counts and the pack kernel
    N, E, R, H = 4, 32, 4, 64
    NT = N * T
    logits = rng.standard_normal((NT, E)).astype(np.float32)
    x = rng.integers(0, 1 << 16, (NT, H), dtype=np.uint16)
    d = Dims(N, T, E, R, H, 0, 0, 0, 0)
    cap = N * T * max(R, E // N)
    sizes = dict(lg=logits.nbytes, x=x.nbytes, ti=4 * NT * R, tw=4 * NT * R, ec=4 * E, eo=4 * (E + 1), rc=4 * N,
                 ro=4 * (N + 1), sc=4 * N * N, pos=4 * NT * R, st=4, px=2 * H * N * cap, ps=4 * N * cap, ws=1 << 20)
    st = np.empty(1, np.int32)
    b = {k: dmalloc(n) for k, n in sizes.items()}
    assert rt.cudaMemset(b["ws"], 0, ctypes.c_size_t(sizes["ws"])) == 0  # zero-filled before first use
    h2d(b["lg"], logits)
    h2d(b["x"], x)
    rc = lib.moe_dispatch_fused(ctypes.byref(d), b["lg"], None, 0, 1, b["x"], None, b["ti"], b["tw"], b["ec"],
                                b["eo"], b["rc"], b["ro"], b["sc"], b["pos"], b["st"], b["px"], None, b["ps"],
                                b["ws"], None)
    assert rc == 0, (rc, lib.moe_last_error())
    assert rt.cudaDeviceSynchronize() == 0
    pos = np.empty((NT, R), np.int32)
    d2h(pos, b["pos"])
    d2h(st, b["st"])
    assert int(st[0]) == 0, int(st[0])
    for p in b.values():
        rt.cudaFree(p)
    return pos

lib.moe_last_error.restype = ctypes.c_char_p
rng = np.random.default_rng(5)
a_pos, a_ec = count_round()
a_small, a_two = fused_round(64), fused_round(256)
assert rt.cudaDeviceReset() == 0
rng = np.random.default_rng(5)
b_pos, b_ec = count_round()
b_small, b_two = fused_round(64), fused_round(256)
assert (a_pos == b_pos).all() and (a_ec == b_ec).all()
assert (a_small == b_small).all() and (a_two == b_two).all()
assert int(a_ec.sum()) == 4 * 1280 * 8
print("RESET_OK")
'''


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()


def test_calls_after_a_device_reset_set_their_attributes_again():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=300)
    assert "RESET_OK" in r.stdout, r.stdout + r.stderr
