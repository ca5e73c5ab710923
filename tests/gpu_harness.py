"""Shared driver for the GPU parity tests: runs one layer through the C ABI
and checks every stage against the float64 oracle on the same inputs.

Inputs come from ``workload`` only; expected values come from ``oracle`` only.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

import sparse_kv_cache_gb300 as skv
from oracle import shadowkv_ref as ref
from workload import Workload, make_A, make_B, make_decode_inputs, make_K_exact, make_V


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def e5m2_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of e5m2 values at |x|: 2^(e-2) in [2^e, 2^(e+1)), 2^-16 below 2^-14."""
    a = np.maximum(np.abs(x), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(a)) - 2)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


# Parity summaries of the run_and_check calls of this session, printed at its end by the
# conftest hook (max output error against the stored-precision oracle and against float64 keys
# that were never stored, the near ties and the hit rates).
REPORTS: list = []


@dataclass
class Report:
    near_ties_sel: int = 0
    near_ties_out: int = 0
    max_out_err: float = 0.0
    max_out_rel: float = 0.0
    max_err_vs_unrounded: float = 0.0   # against float64 keys that were never stored
    steps: int = 0
    alphas: list = field(default_factory=list)


class LayerRun:
    """One layer on the GPU plus lazily computed oracle state per unit."""

    def __init__(self, w: Workload, steps: int, gen_device: str = "cpu", layer: int = 0,
                 side_stream: bool = True, host_alloc: str = "pinned", exact_keys: bool = False):
        self.w, self.steps = w, steps
        dev = torch.device("cuda")
        A = make_A(w, layer, gen_device)
        B = make_B(w, layer, gen_device)
        # pre-filling from exact keys: the library reads them during prefill only
        self.K_src = make_K_exact(w, layer, gen_device, A, B) if exact_keys else None
        V = make_V(w, layer, gen_device)
        q, kn, vn = make_decode_inputs(w, layer, steps, gen_device)
        self.A_d, self.B_d = A.to(dev), B.to(dev)
        if w.v_place == "host" and host_alloc in ("arena", "huge"):
            # page-locked ("arena") or huge-page ("huge") host memory from the library
            self.V_buf = skv.HostBuffer((V.numel() + 64,), V.dtype, kind="huge" if host_alloc == "huge" else "pinned")
            self.V_buf.fill_from(V, 64)
            self.V_arg = self.V_buf.slice(64, V.shape)     # an interior slice, as the bench uses
            self.V_cpu = self.V_arg
        elif w.v_place == "host":
            self.V_arg = V.to("cpu").pin_memory()
            self.V_cpu = self.V_arg
        else:
            self.V_arg = V.to(dev)
            self.V_cpu = None
        self.q_d, self.kn_d, self.vn_d = q.to(dev), kn.to(dev), vn.to(dev)
        self.A_src, self.B_src, self.V_src = A, B, V   # on gen_device, for the oracle
        self.q_src, self.kn_src, self.vn_src = q, kn, vn
        del A, B, V
        self.cfg = skv.make_config(w, max_new_tokens=steps)
        self.main = torch.cuda.Stream()
        self.side = torch.cuda.Stream(priority=-10) if side_stream else None
        self.layer = skv.Layer(self.cfg, self.A_d, self.B_d, self.V_arg, stream=self.main,
                               K=None if self.K_src is None else self.K_src.to(dev))
        self.U, self.G, self.K = w.units, w.group, w.n_select
        self.out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=self.q_d.dtype, device=dev)
        self.sel = torch.empty((w.batch, w.n_kv_heads, w.n_select), dtype=torch.int32, device=dev)
        self.t = 0
        self._pre = {}
        self._anew = {}

    # ------------------------------------------------------------ exports
    def export(self, field: str, dtype, shape):
        n = self.layer.export_size(field)
        elem = torch.empty((), dtype=dtype).element_size()
        buf = torch.empty(n // elem, dtype=dtype, device="cuda")
        self.layer.export(field, buf, stream=self.main)
        self.main.synchronize()
        return buf.view(*shape)

    def sdtype(self):
        """Storage of the keys (and, except in the fp8 configuration, of landmarks and values)."""
        return torch.float32 if self.w.dtype == "f32" else torch.bfloat16

    def vdtype(self):
        """Storage of the values and the landmarks."""
        return torch.float8_e5m2 if self.w.dtype == "fp8" else self.sdtype()

    # ------------------------------------------------------------ oracle per unit
    def unit_inputs(self, u: int):
        b, h = divmod(u, self.w.n_kv_heads)
        return (np64(self.A_src[b]), np64(self.B_src[b, h]), np64(self.V_src[b, h]))

    def oracle_new_state(self, s: int, b: int) -> np.ndarray:
        """ShadowKV+: a = k'.Psi of generated token s of batch element b, in A's storage."""
        key = (s, b)
        if key not in self._anew:
            self._anew[key] = ref.project_new_key(np64(self.kn_src[s, b]), np64(self.B_src[b]),
                                                  ref.key_storage(self.w.dtype))
        return self._anew[key]

    def oracle_prefill(self, u: int) -> ref.UnitPrefill:
        if u not in self._pre:
            A, B, V = self.unit_inputs(u)
            w = self.w
            Kx = None
            if self.K_src is not None:
                b, h = divmod(u, w.n_kv_heads)
                Kx = np64(self.K_src[b, h])
            self._pre[u] = (ref.prefill_unit(A, B, V, w.chunk, w.n_outlier, w.local_window, w.rope_base,
                                             K_exact=Kx), A, B, V)
        return self._pre[u][0]

    # ------------------------------------------------------------ steps
    def enqueue(self):
        """Enqueue the next decode step on the layer's streams without waiting for it."""
        t = self.t
        with torch.cuda.stream(self.main):
            self.layer.decode_step(self.q_d[t], self.kn_d[t], self.vn_d[t], self.out, self.sel,
                                   main=self.main, side=self.side)
        self.t += 1

    def step(self):
        torch.cuda.current_stream().synchronize()
        self.enqueue()
        self.main.synchronize()


def check_prefill(run: LayerRun, units) -> dict:
    """Outliers, chunk ids, landmarks, min-cos, outlier and local K/V of the
    given units against the oracle's Algorithm 1."""
    w = run.w
    U, O, C, W, d = w.units, w.n_outlier, w.chunk, w.local_window, w.head_dim
    ncand = w.n_chunks - W // C
    sd, vd = run.sdtype(), run.vdtype()
    kd = ref.key_storage(w.dtype)
    L_t = run.export("landmarks", vd, (U, w.n_selectable, d))
    ids_t = run.export("chunk_ids", torch.int32, (U, w.n_selectable))
    oid = run.export("outlier_ids", torch.int32, (U, O)).cpu().numpy() if O else np.zeros((U, 0), int)
    mcos_t = run.export("min_cos", torch.float32, (U, ncand))
    kout_t = run.export("k_outlier", sd, (U, O * C, d)) if O else None
    vout_t = run.export("v_outlier", vd, (U, O * C, d)) if O else None
    kloc_t = run.export("k_local", sd, (U, W + run.steps, d))
    vloc_t = run.export("v_local", vd, (U, W + run.steps, d))
    ties = 0
    for u in units:
        pre = run.oracle_prefill(u)
        _, A, B, V = run._pre[u]
        L, mcos, ids = {u: np64(L_t[u])}, {u: np64(mcos_t[u])}, {u: ids_t[u].cpu().numpy()}
        kout = {u: np64(kout_t[u])} if O else None
        vout = {u: np64(vout_t[u])} if O else None
        kloc, vloc = {u: np64(kloc_t[u])}, {u: np64(vloc_t[u])}
        # min-cos per candidate chunk (fp32 arithmetic on exact inputs)
        _within(mcos[u], pre.min_cos, 1e-4, "min-cos")
        # outliers: identical except within the near-tie band of the O-th value
        if O:
            band, _ = ref.near_tie_band(-pre.min_cos, O, 1e-4)
            bs = set(band.tolist())
            g, o = set(oid[u].tolist()), set(pre.outlier_ids.tolist())
            assert len(g) == O and list(oid[u]) == sorted(oid[u])
            assert g - bs == o - bs, f"outliers differ outside the near-tie band (unit {u})"
            ties += len((g ^ o) & bs)
        # chunk ids: the candidates that are not outliers, ascending
        want_ids = np.setdiff1d(np.arange(ncand), oid[u])
        assert np.array_equal(ids[u], want_ids)
        # landmarks of the GPU's chunk ids
        Lo = pre.all_landmarks[ids[u]]
        if w.dtype == "bf16":
            _within(L[u], ref.bf16_round(Lo), bf16_ulp(Lo) + FP32_ABS, "landmarks (bf16)")
        elif w.dtype == "fp8":
            # the GPU rounds its fp32 mean, the oracle its float64 mean: one e5m2 step apart at most
            _within(L[u], ref.e5m2_round(Lo), e5m2_ulp(Lo) + FP32_ABS, "landmarks (e5m2)")
        else:
            _within(L[u], Lo, 2e-5, "landmarks (fp32)")
        # outlier chunks' keys and values
        if O:
            tok = ref.chunk_tokens(oid[u], C)
            Ko = _context_keys(run, u, A, B, tok)
            _close_keys(kout[u], Ko, kd, "k_outlier")
            assert np.array_equal(vout[u], V[tok]), "v_outlier"
        # local window
        Kl = _context_keys(run, u, A, B, np.arange(w.seq_len - W, w.seq_len))
        _close_keys(kloc[u][:W], Kl, kd, "k_local")
        assert np.array_equal(vloc[u][:W], V[w.seq_len - W:]), "v_local"
    return {"outlier_near_ties": ties}


# Absolute floor for values the GPU forms in fp32 before rounding to bf16: the
# rank-r dot products and 8-term means of O(1) keys carry fp32 rounding of a
# few 1e-7; near zero that exceeds one bf16 ulp of the exact value.
FP32_ABS = 1e-5


def _within(gpu: np.ndarray, want: np.ndarray, tol, what: str):
    excess = np.abs(gpu - want) - tol
    if np.any(excess > 0):
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(f"{what}: worst at {i}: gpu {gpu[i]!r} want {want[i]!r} "
                             f"tol {np.broadcast_to(tol, excess.shape)[i]!r} ({int(np.sum(excess > 0))} over)")


def _close_keys(gpu: np.ndarray, want: np.ndarray, dtype: str, what: str):
    assert gpu.shape == want.shape, what
    if want.size == 0:
        return
    if dtype == "bf16":
        _within(gpu, want, bf16_ulp(want) + FP32_ABS, what)
    else:
        _within(gpu, want, 2e-5 * max(1.0, float(np.max(np.abs(want)))), what)


def check_step(run: LayerRun, units, rep: Report, prev_sel: dict, check_cache: bool = True, cache_units=None):
    """After run.step(): selection, hit/miss count, cache slots and output of
    the given units against the oracle on the GPU's state (cache slots of
    ``cache_units`` only, when given)."""
    w = run.w
    t = run.t - 1
    U, G, K, C, d, W = w.units, w.group, w.n_select, w.chunk, w.head_dim, w.local_window
    sd, vd = run.sdtype(), run.vdtype()
    kd = ref.key_storage(w.dtype)
    L_t = run.export("landmarks", vd, (U, w.n_selectable, d))
    ids_t = run.export("chunk_ids", torch.int32, (U, w.n_selectable))
    oid = run.export("outlier_ids", torch.int32, (U, w.n_outlier)).cpu().numpy() if w.n_outlier else None
    sel = run.sel.view(U, K).cpu().numpy()
    exp_sel = run.export("selection", torch.int32, (U, K)).cpu().numpy()
    slots = run.export("slot_of_sel", torch.int32, (U, K)).cpu().numpy()
    mcount = run.export("miss_count", torch.int32, (U,)).cpu().numpy()
    assert np.array_equal(sel, exp_sel), "sel_out and internal selection differ"
    out = np64(run.out).reshape(U, G, d)
    q = np64(run.q_src[t]).reshape(U, G, d)
    kc_t = vc_t = None
    if check_cache:
        kc_t = run.export("k_cache", sd, (U, K * C, d))
        vc_t = run.export("v_cache", vd, (U, K * C, d))
    for u in units:
        pre = run.oracle_prefill(u)
        _, A, B, V = run._pre[u]
        L, ids = {u: np64(L_t[u])}, {u: ids_t[u].cpu().numpy()}
        if check_cache:
            kc, vc = {u: np64(kc_t[u])}, {u: np64(vc_t[u])}
        assert np.all(np.diff(sel[u]) > 0), "selection not ascending"
        assert sorted(slots[u].tolist()) == list(range(K)), "slots not a permutation"
        # selection on the GPU's stored landmarks, scores in float64
        res = ref.select_chunks(q[u], L[u], ids[u], K)
        band, _ = ref.near_tie_band(res["S2"], K, 1e-4)
        bset = set(ids[u][band].tolist())
        g, o = set(sel[u].tolist()), set(res["sel"].tolist())
        assert g - bset == o - bset, f"selection differs outside the near-tie band (unit {u}, step {t})"
        rep.near_ties_sel += len((g ^ o) & bset)
        # hit/miss against the previous step's GPU selection
        hits, misses = ref.hit_miss(prev_sel.get(u), sel[u])
        assert mcount[u] == len(misses), f"miss count (unit {u}, step {t})"
        prev_sel[u] = sel[u].copy()
        # cache slots hold RoPE(A.B) and V of the chunk they claim
        if check_cache and (cache_units is None or u in cache_units):
            for i in range(K):
                ch, s = int(sel[u][i]), int(slots[u][i])
                tok = ref.chunk_tokens([ch], C)
                _close_keys(kc[u][s * C:(s + 1) * C], ref.rebuild_keys(A[tok], B, tok, w.rope_base), kd,
                            "k_cache")
                assert np.array_equal(vc[u][s * C:(s + 1) * C], V[tok]), "v_cache"
        # output = exact attention over the GPU's index set
        b, h = divmod(u, w.n_kv_heads)
        kl = [pre_row for pre_row in _local_keys(run, u, A, B)] + [_new_key(run, s, b, h) for s in range(t + 1)]
        vl = list(V[w.seq_len - W:]) + [np64(run.vn_src[s, b, h]) for s in range(t + 1)]
        oo = oid[u] if oid is not None else []
        ko = _context_keys(run, u, A, B, ref.chunk_tokens(oo, C)) if run.K_src is not None else None
        want = ref.attend_on_index_set(q[u], A, B, V, oo, sel[u], kl, vl, C, w.rope_base, storage=kd,
                                       v_storage=ref.value_storage(w.dtype), k_outlier=ko)
        exact = ref.attend_on_index_set(q[u], A, B, V, oo, sel[u], kl, vl, C, w.rope_base, k_outlier=ko)
        err = np.max(np.abs(out[u] - want))
        rel = err / max(np.max(np.abs(want)), 1e-30)
        rep.max_out_err = max(rep.max_out_err, err)
        rep.max_out_rel = max(rep.max_out_rel, rel)
        rep.max_err_vs_unrounded = max(rep.max_err_vs_unrounded, float(np.max(np.abs(out[u] - exact))))
        if w.dtype in ("bf16", "fp8"):
            assert err <= 2e-2, f"output abs error {err} (unit {u}, step {t})"
        else:
            assert rel <= 1e-4, f"output rel error {rel} (unit {u}, step {t})"
    rep.steps += 1


def _new_key(run: LayerRun, s: int, b: int, h: int) -> np.ndarray:
    """Key of generated token s as attention sees it: as handed in, or (ShadowKV+)
    rebuilt from its rank-r state k'.Psi held in A's storage dtype."""
    w = run.w
    if w.new_keys != "lowrank":
        return np64(run.kn_src[s, b, h])
    a = run.oracle_new_state(s, b)
    return ref.new_token_key(a, np64(run.B_src[b, h]), w.seq_len + s, w.rope_base)


def check_new_states(run: LayerRun, rep_err: list):
    """ShadowKV+: the GPU's rank-r states of the generated tokens so far against
    the oracle's projection, within one storage ulp (fp32 sums against float64)."""
    w = run.w
    t = run.t
    a_t = run.export("a_new", run.sdtype(), (w.batch, run.steps, w.rank))
    for b in range(w.batch):
        for s in range(t):
            want = run.oracle_new_state(s, b)
            got = np64(a_t[b, s])
            tol = (bf16_ulp(want) if w.dtype != "f32" else np.abs(want) * 2.0 ** -22) + 1e-6
            err = np.abs(got - want)
            assert np.all(err <= tol), f"a_new (batch {b}, step {s}): max err {err.max()}"
            rep_err.append(float(err.max()))


def _context_keys(run: LayerRun, u: int, A, B, tok) -> np.ndarray:
    """K_RoPE of context tokens as pre-filling keeps them: the rotated exact keys
    when pre-filling had them, else the factors' keys."""
    w = run.w
    tok = np.asarray(tok, dtype=np.int64)
    if run.K_src is None:
        return ref.rebuild_keys(A[tok], B, tok, w.rope_base)
    b, h = divmod(u, w.n_kv_heads)
    return ref.apply_rope(np64(run.K_src[b, h])[tok], tok, w.rope_base)


def _local_keys(run: LayerRun, u: int, A, B):
    w = run.w
    W = w.local_window
    if W == 0:
        return []
    pos = np.arange(w.seq_len - W, w.seq_len)
    return list(_context_keys(run, u, A, B, pos))


def run_and_check(w: Workload, steps: int, units=None, gen_device="cpu", check_cache=True,
                  side_stream=True, host_alloc="pinned", exact_keys=False, cache_units=None) -> Report:
    run = LayerRun(w, steps, gen_device=gen_device, side_stream=side_stream, host_alloc=host_alloc,
                   exact_keys=exact_keys)
    units = list(range(w.units)) if units is None else list(units)
    check_prefill(run, units)
    rep = Report()
    prev = {}
    a_err = []
    for _ in range(steps):
        run.step()
        check_step(run, units, rep, prev, check_cache=check_cache, cache_units=cache_units)
        if w.new_keys == "lowrank":
            check_new_states(run, a_err)
    st = run.layer.stats()
    assert st["status"] == 0 and st["device_error"] == 0
    assert st["steps"] == steps
    assert st["hits"] + st["misses"] == steps * w.units * w.n_select
    rep.alphas = [st["alpha_mean"], st["alpha_last"]]
    run.layer.close()
    REPORTS.append(summary(w, steps, units, rep, host_alloc if w.v_place == "host" else "hbm"))
    return rep


def summary(w: Workload, steps: int, units, rep: Report, place: str) -> dict:
    return {"workload": f"{w.name} {w.dtype} b{w.batch} S{w.seq_len} G{w.group} {place} drift{w.drift}"
                        + (" plus" if w.new_keys == "lowrank" else ""),
            "steps": steps, "units": len(units), "max_abs": rep.max_out_err, "max_rel": rep.max_out_rel,
            "vs_unrounded": rep.max_err_vs_unrounded, "ties": rep.near_ties_sel,
            "alpha": rep.alphas[0] if rep.alphas else None}
