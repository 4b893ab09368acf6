"""The NVMe expert tier on the host (no GPU): expert slabs replicated over several
files are read into aligned host buffers in two chunks, each read on the replica
expected to finish it first, with the ready bits a device upload would wait on.

Page: "Run Kimi 3.1 locally on one GPU", section "Read the experts the router
needs" (experts on several NVMe drives, O_DIRECT reads into pinned memory,
per-drive concurrency caps, replica choice by expected completion time, decode
fills in two chunks)."""

import os

import numpy as np
import pytest

import moe_synth as syn
from mxfp4_mixture_experts_router_gb300 import binding as B
from mxfp4_mixture_experts_router_gb300 import build as build_mod

TINY = syn.TINY
SLAB = TINY.mxfp4_slab_bytes          # 26,112 bytes
STRIDE = (SLAB + 4095) // 4096 * 4096  # slabs start on 4 KiB boundaries in the files
GU = 2 * (TINY.d_ff * TINY.d_model // 2 + TINY.d_ff * TINY.d_model // 32)


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def _write_store(path, bodies):
    with open(path, "wb") as fh:
        for b, slab in enumerate(bodies):
            fh.write(slab.tobytes())
            fh.write(b"\0" * (STRIDE - SLAB))


def _aligned(n_bytes):
    raw = np.zeros(n_bytes + 4096, dtype=np.uint8)
    off = (-raw.ctypes.data) % 4096
    return raw, raw[off: off + n_bytes]


def test_reads_land_in_two_chunks_on_the_least_loaded_replica(lib, tmp_path):
    bodies = [syn.mxfp4_body_slab(3, b, TINY) for b in range(12)]
    paths = [str(tmp_path / f"drive{i}.bin") for i in range(3)]
    for p in paths:
        _write_store(p, bodies)
    h = B.moe_nvme_open(paths, SLAB, STRIDE, len(bodies), depth=2)
    try:
        keep, buf = _aligned(len(bodies) * STRIDE)
        flags = np.zeros(len(bodies), dtype=np.uint32)
        reps = []
        order = [5, 0, 11, 3, 3, 7, 1, 9, 2, 10, 4, 6, 8]
        for i, b in enumerate(order[:12]):
            dst = buf.ctypes.data + i * STRIDE
            reps.append(B.moe_nvme_read(h, b, dst, GU, flags.ctypes.data + 4 * i))
        for i in range(12):
            assert B.moe_nvme_wait(flags.ctypes.data + 4 * i, B.MOE_SLOT_READY) == B.MOE_OK
            assert flags[i] & B.MOE_SLOT_READY == B.MOE_SLOT_READY and not flags[i] & B.MOE_NVME_FAILED
            got = buf[i * STRIDE: i * STRIDE + SLAB]
            assert np.array_equal(got, bodies[order[i]]), i
        # reads queued back to back spread over the replicas (expected completion time)
        assert len(set(reps)) == 3
        st = [B.moe_nvme_stats(h, r) for r in range(3)]
        assert sum(s["reads"] for s in st) == 12 and sum(s["bytes"] for s in st) == 12 * SLAB
        assert all(s["pending_bytes"] == 0 and s["failures"] == 0 for s in st)
    finally:
        B.moe_nvme_close(h)


def test_first_chunk_bit_comes_before_the_whole_slab(lib, tmp_path):
    bodies = [syn.mxfp4_body_slab(4, b, TINY) for b in range(2)]
    p = str(tmp_path / "drive.bin")
    _write_store(p, bodies)
    h = B.moe_nvme_open([p], SLAB, STRIDE, 2, depth=1)
    try:
        keep, buf = _aligned(STRIDE)
        flag = np.zeros(1, dtype=np.uint32)
        B.moe_nvme_read(h, 1, buf.ctypes.data, GU, flag.ctypes.data)
        assert B.moe_nvme_wait(flag.ctypes.data, B.MOE_SLOT_GATE_UP) == B.MOE_OK
        assert np.array_equal(buf[:GU], bodies[1][:GU])  # the gate/up part is in place
        assert B.moe_nvme_wait(flag.ctypes.data, B.MOE_SLOT_READY) == B.MOE_OK
        assert np.array_equal(buf[:SLAB], bodies[1])
    finally:
        B.moe_nvme_close(h)


def test_a_failed_read_still_sets_its_bits(lib, tmp_path):
    bodies = [syn.mxfp4_body_slab(5, b, TINY) for b in range(3)]
    p = str(tmp_path / "drive.bin")
    _write_store(p, bodies)
    h = B.moe_nvme_open([p], SLAB, STRIDE, 3, depth=1)
    try:
        os.truncate(p, STRIDE)  # the drive loses everything after the first slab
        keep, buf = _aligned(STRIDE)
        flag = np.zeros(1, dtype=np.uint32)
        B.moe_nvme_read(h, 2, buf.ctypes.data, GU, flag.ctypes.data)
        assert B.moe_nvme_wait(flag.ctypes.data, B.MOE_SLOT_READY) == B.MOE_ERR_IO
        assert flag[0] & B.MOE_NVME_FAILED and flag[0] & B.MOE_SLOT_READY == B.MOE_SLOT_READY
        assert B.moe_nvme_stats(h, 0)["failures"] == 1
    finally:
        B.moe_nvme_close(h)


def test_store_shorter_than_its_slabs_is_refused(lib, tmp_path):
    p = str(tmp_path / "short.bin")
    _write_store(p, [syn.mxfp4_body_slab(6, 0, TINY)])
    with pytest.raises(B.MoeError):
        B.moe_nvme_open([p], SLAB, STRIDE, 2, depth=1)
    with pytest.raises(B.MoeError):
        B.moe_nvme_open([str(tmp_path / "missing.bin")], SLAB, STRIDE, 1, depth=1)
