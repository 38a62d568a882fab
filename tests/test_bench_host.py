"""Host logic of bench.py that the JSON line depends on: the whole-job
throughput and the source hash that decides whether stored ncu traffic
still belongs to the current kernel source."""
import os

import bench


def test_job_throughput_counts_every_replica():
    # 4096 tokens per replica, 8 replicas, 0.5 ms per step
    assert bench.job_throughput(4096, 8, 0.5) == 8 * 4096 / 0.5e-3


def _tree(tmp_path, kernel, internal, public):
    csrc = tmp_path / "combine_moe_route_topk_gb300" / "csrc"
    inc = tmp_path / "include"
    csrc.mkdir(parents=True)
    inc.mkdir()
    (csrc / "k.cu").write_text(kernel)
    (csrc / "helpers.cuh").write_text("__device__ int twice(int v) { return 2 * v; }\n")
    (csrc / "moe_internal.cuh").write_text(internal)
    (inc / "moe_route.h").write_text(public)


KERNEL = '#include "helpers.cuh"\n#include "moe_internal.cuh"\n__global__ void k() {}\n'
INTERNAL = '#include "moe_route.h"\nint launch_a(int);\n'
PUBLIC = '#define MOE_OK 0\nint moe_a(void);\n'


def _hash(tmp_path, monkeypatch, kernel=KERNEL, internal=INTERNAL, public=PUBLIC):
    _tree(tmp_path, kernel, internal, public)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return bench.source_hash("k.cu")


def test_source_hash_follows_headers_but_not_declarations(tmp_path, monkeypatch):
    base = _hash(tmp_path / "a", monkeypatch)
    # a new host declaration in either declaration header: same kernel
    assert _hash(tmp_path / "b", monkeypatch, internal=INTERNAL + "int launch_b(int);\n") == base
    assert _hash(tmp_path / "c", monkeypatch, public=PUBLIC + "int moe_b(void);\n") == base
    # the library version is not kernel input either
    assert _hash(tmp_path / "f", monkeypatch, public=PUBLIC + "#define MOE_VERSION 10200\n") == base
    # a changed constant the kernel can see, or a changed kernel line: different
    assert _hash(tmp_path / "d", monkeypatch, public=PUBLIC.replace("MOE_OK 0", "MOE_OK 1")) != base
    assert _hash(tmp_path / "e", monkeypatch, kernel=KERNEL + "// edit\n") != base
