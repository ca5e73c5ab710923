"""ctypes binding of libshadowkv.so (argument marshalling only).

Every step of the decode path runs in the library's CUDA kernels; this module
only turns torch tensors into pointers and streams into handles, and checks
return codes.  There is no fallback: if the library is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libshadowkv.so")

SKV_F32, SKV_BF16, SKV_FP8 = 0, 1, 2
DTYPE_CODES = {"f32": SKV_F32, "bf16": SKV_BF16, "fp8": SKV_FP8}
SKV_V_HBM, SKV_V_HOST = 0, 1
HOST_KINDS = {"pinned": 0, "huge": 1}   # SKV_HOST_PINNED, SKV_HOST_HUGE
PHASES = ("score", "select", "rebuild", "fetch", "attn")
FIELDS = {
    "landmarks": 0, "chunk_ids": 1, "outlier_ids": 2, "min_cos": 3, "k_outlier": 4, "v_outlier": 5,
    "k_local": 6, "v_local": 7, "k_cache": 8, "v_cache": 9, "selection": 10, "slot_of_sel": 11,
    "miss_count": 12, "hits_per_step": 13, "a_new": 14,
}
NEW_KEYS = {"exact": 0, "lowrank": 1}
ERRORS = {0: "OK", -1: "INVALID", -2: "OOM", -3: "NOT_PINNED", -4: "CUDA", -5: "DEVICE_BOUNDS",
          -6: "TIMEOUT", -7: "STEP_LIMIT", -8: "UNSUPPORTED"}
EXPORTED = ("shadowkv_validate_config", "shadowkv_prefill_index", "shadowkv_prefill_index_keys",
            "shadowkv_decode_step",
            "shadowkv_stats", "shadowkv_reset_stats", "shadowkv_set_profiling",
            "shadowkv_set_select_event", "shadowkv_export_size", "shadowkv_export", "shadowkv_model", "shadowkv_destroy",
            "shadowkv_strerror", "shadowkv_version", "shadowkv_host_alloc", "shadowkv_host_alloc_kind",
            "shadowkv_host_repair", "shadowkv_host_free",
            "shadowkv_sparse_attention_noalloc", "shadowkv_sparse_attention_noalloc_status",
            "shadowkv_fetch_probe")


class SkvConfig(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rank", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("n_select", ctypes.c_int32), ("n_outlier", ctypes.c_int32),
                ("local_window", ctypes.c_int32), ("max_new_tokens", ctypes.c_int32),
                ("seq_len", ctypes.c_int64), ("rope_base", ctypes.c_double),
                ("dtype", ctypes.c_int32), ("v_place", ctypes.c_int32),
                ("new_keys", ctypes.c_int32)]


class SkvStats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("units", ctypes.c_int64), ("n_select", ctypes.c_int64),
                ("hits", ctypes.c_int64), ("misses", ctypes.c_int64),
                ("alpha_last", ctypes.c_double), ("alpha_mean", ctypes.c_double),
                ("hbm_bytes", ctypes.c_double), ("link_bytes", ctypes.c_double),
                ("scratch_bytes", ctypes.c_double),
                ("phase_ms", ctypes.c_double * 5), ("phase_launches", ctypes.c_int64 * 5),
                ("device_error", ctypes.c_int32), ("kernel_launches", ctypes.c_int64)]


class SkvAttentionArgs(ctypes.Structure):
    _fields_ = [("units", ctypes.c_int32), ("group", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("n_outlier_tokens", ctypes.c_int32), ("n_cache_tokens", ctypes.c_int32),
                ("n_local_tokens", ctypes.c_int32), ("local_capacity", ctypes.c_int32),
                ("q", ctypes.c_void_p), ("k_outlier", ctypes.c_void_p), ("v_outlier", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("k_local", ctypes.c_void_p),
                ("v_local", ctypes.c_void_p), ("out", ctypes.c_void_p)]


class SkvModel(ctypes.Structure):
    _fields_ = [("eq_bandwidth_gbs", ctypes.c_double), ("memory_savings", ctypes.c_double),
                ("compression_ratio", ctypes.c_double), ("hbm_bytes_per_step", ctypes.c_double),
                ("link_bytes_per_step", ctypes.c_double), ("t_pred_us", ctypes.c_double)]


class ShadowKVError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({strerror(code)})")


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libshadowkv.so (built in-tree by ``sparse_kv_cache_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with sparse_kv_cache_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.shadowkv_validate_config.argtypes = [ctypes.POINTER(SkvConfig)]
    lib.shadowkv_prefill_index.argtypes = [ctypes.POINTER(SkvConfig), vp, vp, vp, vp, ctypes.POINTER(vp)]
    lib.shadowkv_prefill_index_keys.argtypes = [ctypes.POINTER(SkvConfig), vp, vp, vp, vp, vp, ctypes.POINTER(vp)]
    lib.shadowkv_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.shadowkv_stats.argtypes = [vp, ctypes.POINTER(SkvStats)]
    lib.shadowkv_reset_stats.argtypes = [vp]
    lib.shadowkv_set_profiling.argtypes = [vp, i32]
    lib.shadowkv_set_select_event.argtypes = [vp, vp]
    lib.shadowkv_export_size.argtypes = [vp, i32]
    lib.shadowkv_export_size.restype = i64
    lib.shadowkv_export.argtypes = [vp, i32, vp, sz, vp]
    lib.shadowkv_model.argtypes = [ctypes.POINTER(SkvConfig), ctypes.c_double, i64, ctypes.c_double,
                                   ctypes.c_double, ctypes.POINTER(SkvModel)]
    lib.shadowkv_destroy.argtypes = [vp]
    lib.shadowkv_destroy.restype = None
    lib.shadowkv_strerror.argtypes = [i32]
    lib.shadowkv_strerror.restype = ctypes.c_char_p
    lib.shadowkv_version.argtypes = []
    lib.shadowkv_host_alloc.argtypes = [sz, ctypes.POINTER(vp)]
    lib.shadowkv_host_alloc.restype = i32
    lib.shadowkv_host_alloc_kind.argtypes = [sz, i32, ctypes.POINTER(vp)]
    lib.shadowkv_host_alloc_kind.restype = i32
    lib.shadowkv_host_repair.argtypes = [vp, sz]
    lib.shadowkv_host_repair.restype = i32
    lib.shadowkv_host_free.argtypes = [vp]
    lib.shadowkv_host_free.restype = None
    lib.shadowkv_sparse_attention_noalloc.argtypes = [ctypes.POINTER(SkvAttentionArgs), vp]
    lib.shadowkv_sparse_attention_noalloc.restype = i32
    lib.shadowkv_sparse_attention_noalloc_status.argtypes = [vp]
    lib.shadowkv_fetch_probe.argtypes = [vp, sz, i64, i32, ctypes.c_uint64, i32, i32, vp,
                                         ctypes.POINTER(ctypes.c_double)]
    lib.shadowkv_fetch_probe.restype = i32
    lib.shadowkv_sparse_attention_noalloc_status.restype = i32
    for name in ("shadowkv_validate_config", "shadowkv_prefill_index", "shadowkv_decode_step",
                 "shadowkv_stats", "shadowkv_reset_stats", "shadowkv_set_profiling",
                 "shadowkv_set_select_event", "shadowkv_export", "shadowkv_model", "shadowkv_version"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().shadowkv_strerror(code).decode()


def _check(code: int, where: str):
    if code != 0:
        raise ShadowKVError(code, where)


def make_config(w=None, **kw) -> SkvConfig:
    """Config from a ``workload.Workload`` (or keyword fields)."""
    f = {}
    if w is not None:
        f = dict(batch=w.batch, n_kv_heads=w.n_kv_heads, n_q_heads=w.n_q_heads,
                 head_dim=w.head_dim, rank=w.rank, chunk=w.chunk, n_select=w.n_select,
                 n_outlier=w.n_outlier, local_window=w.local_window, max_new_tokens=w.steps,
                 seq_len=w.seq_len, rope_base=w.rope_base,
                 dtype=DTYPE_CODES[w.dtype],
                 v_place=SKV_V_HOST if w.v_place == "host" else SKV_V_HBM,
                 new_keys=NEW_KEYS[w.new_keys])
    f.update(kw)
    return SkvConfig(**f)


def validate_config(cfg: SkvConfig) -> int:
    return load().shadowkv_validate_config(ctypes.byref(cfg))


def model(cfg: SkvConfig, alpha: float, t: int, b_gpu_gbs: float, b_link_gbs: float) -> dict:
    out = SkvModel()
    _check(load().shadowkv_model(ctypes.byref(cfg), alpha, t, b_gpu_gbs, b_link_gbs, ctypes.byref(out)),
           "shadowkv_model")
    return {k: getattr(out, k) for k, _ in SkvModel._fields_}


def sparse_attention_noalloc(q, k_outlier, v_outlier, k_cache, v_cache, k_local, v_local, out,
                             units: int, group: int, n_outlier_tokens: int, n_cache_tokens: int,
                             n_local_tokens: int, local_capacity: int, stream=None) -> int:
    """shadowkv_sparse_attention_noalloc (bf16 tensors); returns the status code."""
    a = SkvAttentionArgs(units=units, group=group, dtype=SKV_BF16, n_outlier_tokens=n_outlier_tokens,
                         n_cache_tokens=n_cache_tokens, n_local_tokens=n_local_tokens,
                         local_capacity=local_capacity, q=_ptr(q), k_outlier=_ptr(k_outlier),
                         v_outlier=_ptr(v_outlier), k_cache=_ptr(k_cache), v_cache=_ptr(v_cache),
                         k_local=_ptr(k_local), v_local=_ptr(v_local), out=_ptr(out))
    return load().shadowkv_sparse_attention_noalloc(ctypes.byref(a), _stream(stream))


def sparse_attention_noalloc_setup(stream=None) -> int:
    """shadowkv_sparse_attention_noalloc with units = 0: the per-device set-up only."""
    a = SkvAttentionArgs(units=0, group=1, dtype=SKV_BF16)
    return load().shadowkv_sparse_attention_noalloc(ctypes.byref(a), _stream(stream))


def sparse_attention_noalloc_status(stream=None) -> int:
    """shadowkv_sparse_attention_noalloc_status: the kept kernel status, cleared on read."""
    return load().shadowkv_sparse_attention_noalloc_status(_stream(stream))


def fetch_probe(src_ptr: int, nbytes: int, n_chunks: int, chunk_bytes: int = 2048, seed: int = 1,
                reps: int = 3, fresh: bool = False, stream=None) -> float:
    """shadowkv_fetch_probe: GB/s of the fetch kernel on random chunks of [src, src + nbytes)
    (fresh: new chunks for every repetition)."""
    g = ctypes.c_double()
    _check(load().shadowkv_fetch_probe(src_ptr, nbytes, n_chunks, chunk_bytes, seed, reps, 1 if fresh else 0,
                                       _stream(stream), ctypes.byref(g)), "shadowkv_fetch_probe")
    return g.value


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


class HostBuffer:
    """Host memory for values from shadowkv_host_alloc_kind, viewed as a CPU tensor:
    kind "pinned" (page-locked) or "huge" (transparent huge pages read through the
    host's page tables)."""

    def __init__(self, shape, dtype, kind: str = "pinned"):
        import numpy as np
        import torch
        self.shape, self.dtype, self.kind = tuple(shape), dtype, kind
        elem = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(self.shape)) * elem
        p = ctypes.c_void_p()
        _check(load().shadowkv_host_alloc_kind(self.nbytes, HOST_KINDS[kind], ctypes.byref(p)),
               "shadowkv_host_alloc_kind")
        self._p = p
        raw = (ctypes.c_uint8 * self.nbytes).from_address(p.value)
        self.tensor = torch.frombuffer(raw, dtype=torch.uint8).view(dtype).view(self.shape)

    def data_ptr(self) -> int:
        return self._p.value

    def fill_from(self, src, offset_elems: int = 0):
        """Copy a tensor (any device) into the buffer starting at element offset_elems."""
        flat = self.tensor.view(-1)
        s = src.contiguous().view(-1)
        flat[offset_elems:offset_elems + s.numel()].copy_(s)

    def repair(self) -> int:
        """shadowkv_host_repair over the whole buffer (huge-page kind); returns the status."""
        return load().shadowkv_host_repair(self._p, self.nbytes)

    def slice(self, offset_elems: int, shape):
        """A view of part of the buffer (data_ptr() gives its address)."""
        import numpy as np
        n = int(np.prod(shape))
        return self.tensor.view(-1)[offset_elems:offset_elems + n].view(*shape)

    def free(self):
        if getattr(self, "_p", None) and self._p.value:
            self.tensor = None
            load().shadowkv_host_free(self._p)
            self._p = ctypes.c_void_p()

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class Layer:
    """One layer's ShadowKV state (the handle of shadowkv_prefill_index)."""

    def __init__(self, cfg: SkvConfig, A, B, V, stream=None, K=None):
        """K: optional exact pre-RoPE keys [b][H][S][d] (pre-filling from exact keys)."""
        lib = load()
        self.cfg = cfg
        self._keep = (A, B, V)   # the library borrows these
        h = ctypes.c_void_p()
        if K is None:
            _check(lib.shadowkv_prefill_index(ctypes.byref(cfg), _ptr(A), _ptr(B), _ptr(V), _stream(stream),
                                              ctypes.byref(h)), "shadowkv_prefill_index")
        else:
            _check(lib.shadowkv_prefill_index_keys(ctypes.byref(cfg), _ptr(A), _ptr(B), _ptr(K), _ptr(V),
                                                   _stream(stream), ctypes.byref(h)),
                   "shadowkv_prefill_index_keys")
        self._h = h

    @property
    def handle(self) -> int:
        return self._h.value

    def decode_step(self, q, k_new, v_new, out, sel_out=None, main=None, side=None):
        _check(load().shadowkv_decode_step(self._h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                           _ptr(sel_out), _stream(main),
                                           None if side is None else _stream(side)),
               "shadowkv_decode_step")

    def decode_step_raw(self, q, k_new, v_new, out, sel_out, main, side) -> int:
        """Same call with integer pointers/handles; returns the status code."""
        return load().shadowkv_decode_step(self._h, q, k_new, v_new, out, sel_out, main, side)

    def stats(self, check: bool = True) -> dict:
        s = SkvStats()
        rc = load().shadowkv_stats(self._h, ctypes.byref(s))
        if check:
            _check(rc, "shadowkv_stats")
        d = {k: getattr(s, k) for k, _ in SkvStats._fields_ if k not in ("phase_ms", "phase_launches")}
        d["phase_ms"] = dict(zip(PHASES, list(s.phase_ms)))
        d["phase_launches"] = dict(zip(PHASES, list(s.phase_launches)))
        d["status"] = rc
        return d

    def reset_stats(self):
        _check(load().shadowkv_reset_stats(self._h), "shadowkv_reset_stats")

    def set_profiling(self, on: bool):
        _check(load().shadowkv_set_profiling(self._h, 1 if on else 0), "shadowkv_set_profiling")

    def set_select_event(self, event):
        """Record ``event`` (a torch.cuda.Event, or None to stop) after each step's selection."""
        if event is not None and not event.cuda_event:
            import torch
            event.record(torch.cuda.current_stream())   # torch creates its events on first record
        _check(load().shadowkv_set_select_event(self._h, None if event is None else event.cuda_event),
               "shadowkv_set_select_event")

    def export_size(self, field: str) -> int:
        return load().shadowkv_export_size(self._h, FIELDS[field])

    def export(self, field: str, dst, stream=None):
        _check(load().shadowkv_export(self._h, FIELDS[field], _ptr(dst),
                                      dst.numel() * dst.element_size(), _stream(stream)),
               f"shadowkv_export({field})")

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            load().shadowkv_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
