"""Error behaviour of the C ABI on a GPU, without faulting the GPU: every bad
input is refused on the host with its status code, and nothing leaks."""
import ctypes
import os

import pytest
import torch

import sparse_kv_cache_gb300 as skv
from sparse_kv_cache_gb300 import _binding
from workload import TINY, make_A, make_B, make_V

pytestmark = pytest.mark.gpu

W = TINY.with_(seq_len=1024, n_select=8, n_outlier=2, spike_chunks=2, steps=2)


def _inputs(dev="cuda"):
    return make_A(W, 0).to(dev), make_B(W, 0).to(dev), make_V(W, 0).to(dev)


def _prefill(cfg, A, B, V):
    lib = skv.load()
    h = ctypes.c_void_p()
    rc = lib.shadowkv_prefill_index(ctypes.byref(cfg), A.data_ptr(), B.data_ptr(), V.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream, ctypes.byref(h))
    return rc, h


def test_invalid_config_and_pointers():
    A, B, V = _inputs()
    cfg = skv.make_config(W)
    bad = skv.make_config(W, n_select=10_000)
    assert _prefill(bad, A, B, V)[0] == -1
    # A in host memory while the kernels read it on the device
    assert _prefill(cfg, A.cpu(), B, V)[0] == -1
    # values declared in HBM but given as host memory
    assert _prefill(cfg, A, B, V.cpu().pin_memory())[0] == -1
    # misaligned pointer
    lib = skv.load()
    h = ctypes.c_void_p()
    rc = lib.shadowkv_prefill_index(ctypes.byref(cfg), A.data_ptr() + 2, B.data_ptr(), V.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream, ctypes.byref(h))
    assert rc == -1 and not h.value


def test_host_values_reachable_or_refused():
    A, B, V = _inputs()
    cfg = skv.make_config(W, v_place=skv.SKV_V_HOST)
    pageable = V.cpu()
    rc, h = _prefill(cfg, A, B, pageable)
    # page-locked memory is required unless the GPU reads pageable memory through the host page tables
    assert rc in (0, -3)
    if rc == 0:
        skv.load().shadowkv_destroy(h)
    rc, h = _prefill(cfg, A, B, pageable.pin_memory())
    assert rc == 0
    skv.load().shadowkv_destroy(h)


def test_forced_allocation_failure_frees_everything():
    A, B, V = _inputs()
    cfg = skv.make_config(W)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    os.environ["SHADOWKV_FAULT"] = "oom:5"
    try:
        rc, h = _prefill(cfg, A, B, V)
    finally:
        del os.environ["SHADOWKV_FAULT"]
    assert rc == -2 and not h.value
    torch.cuda.synchronize()
    assert abs(torch.cuda.mem_get_info()[0] - free0) < (64 << 20)


def test_step_limit_and_clean_destroy():
    A, B, V = _inputs()
    layer = skv.Layer(skv.make_config(W, max_new_tokens=2), A, B, V)
    q = torch.randn((W.batch, W.n_q_heads, 128), device="cuda")
    kv = torch.randn((W.batch, W.n_kv_heads, 128), device="cuda")
    out = torch.empty_like(q)
    layer.decode_step(q, kv, kv, out)
    layer.decode_step(q, kv, kv, out)
    with pytest.raises(skv.ShadowKVError) as e:
        layer.decode_step(q, kv, kv, out)
    assert e.value.code == -7
    st = layer.stats()
    assert st["steps"] == 2 and st["device_error"] == 0
    layer.close()
    layer.close()                      # a second close is a no-op
    skv.load().shadowkv_destroy(None)  # destroying NULL is allowed


def test_export_checks_buffer_size():
    A, B, V = _inputs()
    layer = skv.Layer(skv.make_config(W), A, B, V)
    small = torch.empty(4, dtype=torch.int32, device="cuda")
    with pytest.raises(skv.ShadowKVError):
        layer.export("chunk_ids", small)
    layer.close()
