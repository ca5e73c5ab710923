"""The C ABI without a GPU: the library builds, loads and exports every symbol
include/shadowkv.h declares; host-only calls (config checks, error strings,
analytical models) behave as specified."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from oracle import shadowkv_ref as ref
from workload import ALL, LLAMA_128K, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "shadowkv.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_kv_cache_gb300 import _binding, build
    if not os.path.exists(_binding.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build the library")
        build.build()
    return _binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(shadowkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("shadowkv_prefill_index", "shadowkv_decode_step", "shadowkv_stats", "shadowkv_destroy",
              "shadowkv_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = lib.load()
    for n in declared_functions():
        assert hasattr(so, n), n
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True).stdout
        exported = set(re.findall(r"\bT (shadowkv_\w+)", out))
        assert set(declared_functions()) <= exported
    assert set(lib.EXPORTED) == set(declared_functions())


def test_struct_layouts_match_header(lib):
    # sizes of the ABI structs as the C compiler lays them out
    src = os.path.join(ROOT, "include", "shadowkv.h")
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc missing")
    prog = ('#include "shadowkv.h"\n#include <stdio.h>\n#include <stddef.h>\n'
            'int main(){printf("%zu %zu %zu %zu %zu\\n", sizeof(skv_config), sizeof(skv_stats), '
            'sizeof(skv_model), offsetof(skv_stats, device_error), sizeof(skv_attention_args));return 0;}\n')
    tmp = os.path.join(ROOT, "sparse_kv_cache_gb300", "_build")
    os.makedirs(tmp, exist_ok=True)
    c = os.path.join(tmp, "abi_sizes.c")
    exe = os.path.join(tmp, "abi_sizes")
    open(c, "w").write(prog)
    subprocess.run([gcc, "-I", os.path.dirname(src), c, "-o", exe], check=True)
    sizes = [int(x) for x in subprocess.run([exe], capture_output=True, text=True).stdout.split()]
    assert sizes == [ctypes.sizeof(lib.SkvConfig), ctypes.sizeof(lib.SkvStats), ctypes.sizeof(lib.SkvModel),
                     lib.SkvStats.device_error.offset, ctypes.sizeof(lib.SkvAttentionArgs)]


def test_strerror_and_version(lib):
    assert lib.strerror(0) == "ok"
    for code in range(-8, 0):
        assert lib.strerror(code) not in ("ok", "unknown error")
    assert lib.load().shadowkv_version() >= 10000


@pytest.mark.parametrize("name", sorted(ALL))
def test_workload_configs_validate(lib, name):
    assert lib.validate_config(lib.make_config(ALL[name])) == 0


@pytest.mark.parametrize("field,value", [
    ("head_dim", 64), ("chunk", 16), ("rank", 12), ("rank", 264), ("n_q_heads", 12), ("n_q_heads", 48),
    ("seq_len", 4100), ("local_window", 12), ("n_select", 0), ("n_select", 5000), ("n_outlier", -1),
    ("max_new_tokens", 0), ("dtype", 3), ("v_place", 2), ("rope_base", 0.5), ("new_keys", 2),
    ("new_keys", -1)])
def test_invalid_configs_rejected(lib, field, value):
    cfg = lib.make_config(TINY)
    setattr(cfg, field, value)
    assert lib.validate_config(cfg) == -1


def test_lowrank_new_keys_config_accepted(lib):
    cfg = lib.make_config(TINY.with_(new_keys="lowrank"))
    assert cfg.new_keys == 1 and lib.validate_config(cfg) == 0


def test_budget_larger_than_selectable_rejected(lib):
    cfg = lib.make_config(TINY)
    cfg.n_select = TINY.n_selectable + 1
    assert lib.validate_config(cfg) == -1
    cfg.n_select = TINY.n_selectable
    assert lib.validate_config(cfg) == 0


@pytest.mark.parametrize("alpha", [0.0, 0.6, 0.9, 1.0])
def test_library_models_match_oracle(lib, alpha):
    w = LLAMA_128K
    cfg = lib.make_config(w)
    m = lib.model(cfg, alpha, 0, 2000.0, 31.5)
    want = ref.equivalent_bandwidth(w.seq_len, w.chunk, w.n_select, w.n_outlier, alpha, 2000.0, 31.5)
    assert abs(m["eq_bandwidth_gbs"] - want) <= 1e-9 * want
    assert abs(m["memory_savings"] - ref.memory_savings(w.seq_len, w.head_dim * w.n_kv_heads, w.chunk,
                                                        w.n_select, w.n_outlier, w.rank)) < 1e-12
    assert abs(m["compression_ratio"] - ref.compression_ratio(w.seq_len, w.head_dim * w.n_kv_heads,
                                                              w.rank)) < 1e-12
    assert m["hbm_bytes_per_step"] > 0 and m["t_pred_us"] > 0


def test_model_reproduces_pages_example(lib):
    # page numbers: 7.2 TB/s at S=128K, C=8, K=256, O=48, alpha=0.6, 2 TB/s, 31.5 GB/s; 7.08x savings
    cfg = lib.make_config(LLAMA_128K)
    m = lib.model(cfg, 0.6, 0, 2000.0, 31.5)
    assert abs(m["eq_bandwidth_gbs"] / 1000 - 7.2) < 0.05
    assert abs(m["memory_savings"] - 7.08) < 0.005


def test_step_bytes_match_the_byte_model_by_hand(lib):
    # the per-unit byte model worked by hand: about 12.66 GB per 32-layer step at 128K,
    # batch 8, alpha 0.6, t = 32 (bf16)
    cfg = lib.make_config(LLAMA_128K)
    m = lib.model(cfg, 0.6, 32, 8000.0, 400.0)
    per_step = 32 * (m["hbm_bytes_per_step"])
    assert 12.0e9 < per_step < 13.2e9


def test_step_bytes_by_value_placement(lib):
    # the missed chunks' values: over the link with host values; with values in HBM the
    # tensor-core path's attention reads them where they live (no slot write, no extra read),
    # while the fp32 path copies them into the value cache (one more read)
    w = LLAMA_128K
    U, C, d, K = w.units, w.chunk, w.head_dim, w.n_select
    misses = 0.4 * K * U
    host = lib.model(lib.make_config(w), 0.6, 32, 8000.0, 400.0)
    hbm = lib.model(lib.make_config(w.with_(v_place="hbm")), 0.6, 32, 8000.0, 400.0)
    assert host["link_bytes_per_step"] == pytest.approx(misses * C * d * 2)
    assert hbm["link_bytes_per_step"] == 0
    assert hbm["hbm_bytes_per_step"] == pytest.approx(host["hbm_bytes_per_step"] - misses * C * d * 2)
    f32 = w.with_(dtype="f32")
    h32 = lib.model(lib.make_config(f32), 0.6, 32, 8000.0, 400.0)
    d32 = lib.model(lib.make_config(f32.with_(v_place="hbm")), 0.6, 32, 8000.0, 400.0)
    assert d32["hbm_bytes_per_step"] == pytest.approx(h32["hbm_bytes_per_step"] + h32["link_bytes_per_step"])
