"""The decode step's value fetch beyond the bf16 cases of the parity file.

* fp32 values in page-locked host memory: the fetch moves 4 KB chunks, eight 16-byte words
  per lane and chunk, two chunks per warp; the slots are checked bit-exact against the host
  rows every step and the outputs against the oracle.
* The fetch-rate probe (shadowkv_fetch_probe), which times the same kernel on random chunks:
  it reports a positive rate for every chunk size, from device and from page-locked host
  memory, warm and fresh, and refuses bad arguments on the host before anything runs.
"""
import pytest
import torch

import sparse_kv_cache_gb300 as skv
from tests.gpu_harness import run_and_check
from workload import TINY

pytestmark = pytest.mark.gpu


def test_tiny_fp32_host_values():
    run_and_check(TINY.with_(v_place="host", seed=9), 4)


def test_fetch_probe_device_and_host_memory():
    dev = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    for cb in (1024, 2048, 4096):
        assert skv.fetch_probe(dev.data_ptr(), dev.numel(), 1000, chunk_bytes=cb, reps=2) > 0
    assert skv.fetch_probe(dev.data_ptr(), dev.numel(), 1000, reps=2, fresh=True) > 0
    host = skv.HostBuffer((64 << 20,), torch.uint8)
    try:
        assert skv.fetch_probe(host.data_ptr(), 64 << 20, 2000, reps=2) > 0
    finally:
        host.free()


def test_fetch_probe_refusals():
    dev = torch.empty(8 << 20, dtype=torch.uint8, device="cuda")
    p, n = dev.data_ptr(), dev.numel()
    bad = [
        dict(src=p, nbytes=n, n_chunks=1000, chunk_bytes=1000),       # not a chunk size
        dict(src=p + 8, nbytes=n - 8, n_chunks=1000, chunk_bytes=2048),  # not 16-byte aligned
        dict(src=p, nbytes=2048 * 1500, n_chunks=1000, chunk_bytes=2048),  # under two slots per chunk
        dict(src=p, nbytes=n, n_chunks=0, chunk_bytes=2048),           # no chunks
    ]
    for a in bad:
        with pytest.raises(skv.ShadowKVError) as e:
            skv.fetch_probe(a["src"], a["nbytes"], a["n_chunks"], chunk_bytes=a["chunk_bytes"], reps=1)
        assert e.value.code == -1, a
