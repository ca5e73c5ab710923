"""Decode-step benchmark of the ShadowKV sparse-attention path on GB300.

One step = one decode step of every layer (all rows of the hot path: landmark
scoring, top-K + index scan + append, key rebuild, value fetch, sparse
attention) for the whole batch.  Default workload: Llama-3.1-8B attention
shape at 128K context, batch 8, 32 layers, values in page-locked host memory.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
of the workload (independent batches, no collective on the data path) and the
timing is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workload import ALL, LLAMA_128K, Workload  # noqa: E402

# DRAM traffic of one scorer launch from ncu captures (dram__bytes_read.sum +
# dram__bytes_write.sum), valid only while the scorer source is the one that was profiled;
# per unit, scaled to a launch by its units.  bf16: k_score_tc at 128K b4 (32 units),
# 133.89 + 4.35 MB; fp8: k_score_f8 at 128K b8 (64 units), 133.94 + 5.40 MB.
SCORE_TRAFFIC_SHA256 = "6b81a89c450e7c0b18c603f24db0192aae24ae37004b7445e69bd0cdc73c951f"
SCORE_TRAFFIC = {
    "bf16": {"seq_len": 131072, "bytes_per_unit": (133885696 + 4347136) / 32},
    "fp8": {"seq_len": 131072, "bytes_per_unit": (133939712 + 5395456) / 64},
}


METRIC = "sparse decode-attention tokens/s and HBM GB/s (% of 8 TB/s) at 128K, 1×GB300"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=LLAMA_128K.name, choices=sorted(ALL))
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count")
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--v-place", default="", choices=["", "hbm", "host"])
    ap.add_argument("--dtype", default="", choices=["", "bf16", "fp8"],
                    help="storage: bf16, or fp8 (e5m2 landmarks and values, bf16 keys and factors)")
    ap.add_argument("--new-keys", default="", choices=["", "exact", "lowrank"],
                    help="lowrank: ShadowKV+ (generated tokens' keys kept at rank r and rebuilt each step)")
    ap.add_argument("--drift", type=float, default=-1.0)
    ap.add_argument("--share-storage", default="auto", choices=["auto", "yes", "no"],
                    help="reuse one layer's A/B/V for every layer (state stays per layer)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=0.0,
                    help="--impl reference: oracle seconds per timed step (default: the run fits in ~2 minutes)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--microbatches", type=int, default=1,
                    help="split the batch into this many handles per layer, each on its own stream pair")
    ap.add_argument("--host-mem", default="pinned", choices=["pinned", "huge"],
                    help="host values: page-locked memory, or transparent huge pages read through the host page tables")
    ap.add_argument("--single-stream", action="store_true",
                    help="run the value fetch on the main stream too (per-kernel timing without overlap)")
    return ap.parse_args()


def workload_from(args) -> Workload:
    w = ALL[args.config]
    kw = {}
    if args.layers:
        kw["layers"] = args.layers
    if args.batch:
        kw["batch"] = args.batch
    if args.v_place:
        kw["v_place"] = args.v_place
    if args.dtype:
        kw["dtype"] = args.dtype
        if args.dtype == "fp8":
            kw["name"] = w.name + "-fp8"
    if args.drift >= 0:
        kw["drift"] = args.drift
    if args.new_keys:
        kw["new_keys"] = args.new_keys
        if args.new_keys == "lowrank":
            kw["name"] = kw.get("name", w.name) + "-plus"
    return w.with_(**kw) if kw else w


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The maximum of a per-rank value over all ranks (identity on one rank)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(base: int, rank: int) -> int:
    """Each rank runs its own independent replica of the workload."""
    return base + 1000 * rank


def score_traffic_per_launch(w: Workload):
    """Measured DRAM bytes per scorer launch, or None once the scorer or the shape differ."""
    import hashlib
    src = os.path.join(ROOT, "sparse_kv_cache_gb300", "csrc", "k_score.cu")
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    t = SCORE_TRAFFIC.get(w.dtype)
    if digest != SCORE_TRAFFIC_SHA256 or t is None or w.seq_len != t["seq_len"]:
        return None
    return t["bytes_per_unit"] * w.units


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def thp_counters() -> dict:
    """Huge-page split and migration counters of the host kernel (/proc/vmstat)."""
    keys = ("thp_split_pmd", "thp_split_page", "thp_fault_alloc", "pgmigrate_success")
    out = {}
    try:
        for line in open("/proc/vmstat"):
            k, _, v = line.partition(" ")
            if k in keys:
                out[k] = int(v)
    except OSError:
        pass
    return out


def mem_available_gb() -> float:
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) / 1e6
    except OSError:
        pass
    return 0.0


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clocks and throttle reasons during a timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.proc, self.path = gpu, None, None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        os.unlink(self.path)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm
def run_ours(args, w: Workload, ws: int, rank: int, local: int):
    import torch
    import torch.distributed as dist

    import sparse_kv_cache_gb300 as skv
    from workload import make_A, make_B, make_decode_inputs, make_V, storage_dtype, value_dtype

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    K, W = args.steps, args.warmup
    passes = 3
    total_steps = W + passes * K
    w = w.with_(seed=replica_seed(w.seed, rank), steps=total_steps)
    L = w.layers
    dt, vdt = storage_dtype(w), value_dtype(w)   # keys, factors, q, out / values
    es = 4 if w.dtype == "f32" else 2
    es_v = 1 if w.dtype == "fp8" else es          # values and landmarks
    v_bytes = w.batch * w.n_kv_heads * w.seq_len * w.head_dim * es_v
    share = args.share_storage == "yes"
    if args.share_storage == "auto" and w.v_place == "host":
        share = mem_available_gb() < 1.3 * L * v_bytes / 1e9 + 16
    n_data = 1 if share else L

    thp0 = thp_counters()
    M = max(1, args.microbatches)
    if w.batch % M:
        raise SystemExit(f"batch {w.batch} is not a multiple of --microbatches {M}")
    bm = w.batch // M
    arena = None
    if w.v_place == "host":
        # one page-locked arena for every layer's values (large allocations keep GPU translations few)
        per = w.batch * w.n_kv_heads * w.seq_len * w.head_dim
        arena = skv.HostBuffer((n_data * per,), vdt, kind=args.host_mem)
    # one (main, side) stream pair per micro-batch; the value fetch (link-bound) goes first
    mains = [torch.cuda.Stream(dev) for _ in range(M)]
    sides = [torch.cuda.Stream(dev, priority=-10) for _ in range(M)]
    main = mains[0]
    data, layers = [], []
    t0 = time.time()
    for ell in range(n_data):
        A = make_A(w, ell, dev)
        B = make_B(w, ell, dev)
        Vd = make_V(w, ell, dev)
        if w.v_place == "host":
            # values stay in host memory; the GPU reads missed chunks in place over NVLink-C2C
            arena.fill_from(Vd, ell * Vd.numel())
            V = arena.slice(ell * Vd.numel(), Vd.shape)
            del Vd
        else:
            V = Vd
        data.append((A, B, V))
    # micro-batch m owns batch rows [m*bm, (m+1)*bm) of every tensor (all are batch-major)
    cfg = skv.make_config(w.with_(batch=bm), max_new_tokens=total_steps)
    for ell in range(L):
        A, B, V = data[ell % n_data]
        for m in range(M):
            rows = slice(m * bm, (m + 1) * bm)
            layers.append(skv.Layer(cfg, A[rows], B[rows], V[rows], stream=main))
    torch.cuda.synchronize()
    setup_s = time.time() - t0

    # per-layer decode inputs for every step, resident in HBM
    qs, kns, vns = [], [], []
    for ell in range(L):
        q, kn, vn = make_decode_inputs(w, ell, total_steps, dev)
        qs.append(q); kns.append(kn); vns.append(vn)
    out = [torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=dt, device=dev) for _ in range(L)]
    hq = [lay.handle for lay in layers]
    lib = skv.load()
    ms_ = [st.cuda_stream for st in mains]
    ss_ = [None if args.single_stream else st.cuda_stream for st in sides]

    def step(s: int):
        # layer order is kept within each micro-batch's stream; the micro-batches run side by side
        for ell in range(L):
            for m in range(M):
                rows = slice(m * bm, (m + 1) * bm)
                rc = lib.shadowkv_decode_step(hq[ell * M + m], qs[ell][s][rows].data_ptr(),
                                              kns[ell][s][rows].data_ptr(), vns[ell][s][rows].data_ptr(),
                                              out[ell][rows].data_ptr(), None, ms_[m], ss_[m])
                if rc:
                    raise skv.ShadowKVError(rc, "decode_step")

    def fork(ev):
        for st in mains[1:]:
            st.wait_event(ev)

    def join():
        for st in mains[1:]:
            ev = torch.cuda.Event()
            ev.record(st)
            main.wait_event(ev)

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    s_idx = 0
    for _ in range(W):
        step(s_idx); s_idx += 1
    for lay in layers:
        lay.reset_stats()

    # ---- pass 1: device-resident inputs (the headline value)
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    fork(e0)
    for _ in range(K):
        step(s_idx); s_idx += 1
    join()
    e1.record(main)
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    st = [lay.stats() for lay in layers]
    hbm = sum(s["hbm_bytes"] for s in st)
    link = sum(s["link_bytes"] for s in st)
    scratch = sum(s["scratch_bytes"] for s in st)
    alpha = statistics.mean(s["alpha_mean"] for s in st)
    # kernels the library launched in the timed steps (its own count per decode step)
    launches = int(sum(s["kernel_launches"] for s in st))

    # ---- pass 2: the same steps with per-phase CUDA events (roofline of the dominant kernel)
    for lay in layers:
        lay.reset_stats()
        lay.set_profiling(True)
    barrier()
    for _ in range(K):
        step(s_idx); s_idx += 1
    barrier()
    st2 = [lay.stats() for lay in layers]
    for lay in layers:
        lay.set_profiling(False)
    phase_ms = {ph: sum(s["phase_ms"][ph] for s in st2) for ph in skv.PHASES}
    phase_n = {ph: sum(s["phase_launches"][ph] for s in st2) for ph in skv.PHASES}
    score_us = 1000.0 * phase_ms["score"] / max(1, phase_n["score"])
    # one scorer launch covers one micro-batch: landmarks + queries of its units
    score_bytes = (w.units // M) * (w.n_selectable * es_v + w.group * es) * w.head_dim
    achieved = score_bytes / (score_us * 1e-6) / 1e9
    score_traffic = score_traffic_per_launch(w.with_(batch=bm))
    peak, peak_kind = measured_peaks()

    # ---- pass 3: end to end through the public call with host buffers.  Every step copies
    # its inputs (q, k_new, v_new of every layer, packed in one page-locked buffer) to the
    # device in one copy and reads every layer's output back in one copy, both on a copy
    # stream; the device buffers are double-buffered so the next step's inputs arrive while
    # this step computes.  The timed region holds all K steps' copies.
    e2e = None
    if not args.no_e2e:
        nq, nk, nv = qs[0][0].numel(), kns[0][0].numel(), vns[0][0].numel()
        per_layer = nq + nk + nv
        hin = torch.empty((K, L, per_layer), dtype=dt, pin_memory=True)
        for k in range(K):
            for ell in range(L):
                hin[k, ell, :nq].copy_(qs[ell][s_idx + k].reshape(-1))
                hin[k, ell, nq:nq + nk].copy_(kns[ell][s_idx + k].reshape(-1))
                hin[k, ell, nq + nk:].copy_(vns[ell][s_idx + k].reshape(-1))
        din = [torch.empty((L, per_layer), dtype=dt, device=dev) for _ in range(2)]
        dout = [torch.empty((L,) + tuple(out[0].shape), dtype=dt, device=dev) for _ in range(2)]
        hout = torch.empty((K, L) + tuple(out[0].shape), dtype=dt, pin_memory=True)
        cs = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(K)]
        ev_done = [torch.cuda.Event() for _ in range(K)]     # step k's kernels finished (main)
        ev_read = [torch.cuda.Event() for _ in range(K)]     # step k's outputs copied back (cs)
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(main)
        fork(f0)
        cs.wait_event(f0)

        def upload(k):
            if k >= 2:
                cs.wait_event(ev_done[k - 2])                # din[k % 2] is free again
            with torch.cuda.stream(cs):
                din[k % 2].copy_(hin[k], non_blocking=True)
            ev_in[k].record(cs)

        upload(0)
        for k in range(K):
            if k + 1 < K:
                upload(k + 1)
            b_in, b_out = din[k % 2], dout[k % 2]
            for m in range(M):
                mains[m].wait_event(ev_in[k])
                if k >= 2:
                    mains[m].wait_event(ev_read[k - 2])      # dout[k % 2] was read back
            for ell in range(L):
                qv = b_in[ell, :nq].view(qs[ell][0].shape)
                kv = b_in[ell, nq:nq + nk].view(kns[ell][0].shape)
                vv = b_in[ell, nq + nk:].view(vns[ell][0].shape)
                for m in range(M):
                    rows = slice(m * bm, (m + 1) * bm)
                    layers[ell * M + m].decode_step(qv[rows], kv[rows], vv[rows], b_out[ell][rows], None,
                                                    main=mains[m],
                                                    side=None if args.single_stream else sides[m])
            for m in range(1, M):
                ev = torch.cuda.Event()
                ev.record(mains[m])
                main.wait_event(ev)
            ev_done[k].record(main)
            cs.wait_event(ev_done[k])
            with torch.cuda.stream(cs):
                hout[k].copy_(b_out, non_blocking=True)
            ev_read[k].record(cs)
        main.wait_event(ev_read[K - 1])
        join()
        f1.record(main)
        barrier()
        ms_e2e = max_over_ranks(f0.elapsed_time(f1), ws, dev)
        h2d = L * per_layer * es
        d2h = L * out[0].numel() * es
        e2e = {"value": ws * w.batch * K / (ms_e2e / 1000.0), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        s_idx += K

    # host-link bandwidth, measured live: page-locked host -> HBM copy of 256 MB from the value arena
    b_link = None
    if arena is not None:
        n = min(arena.tensor.numel(), (256 << 20) // es_v)
        dbuf = torch.empty(n, dtype=vdt, device=dev)
        src = arena.tensor.view(-1)[:n]
        dbuf.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(3):
            dbuf.copy_(src, non_blocking=True)
        c1.record()
        torch.cuda.synchronize()
        b_link = 3 * n * es_v / (c0.elapsed_time(c1) * 1e-3) / 1e9
        del dbuf
    # the pages' equivalent-bandwidth model with the measured hit rate and bandwidths: predicted step time
    peak_gbs, _ = measured_peaks()
    cfg_m = skv.make_config(w, max_new_tokens=total_steps)
    t_mid = W + K // 2
    mdl = skv.model(cfg_m, max(0.0, min(1.0, alpha)), t_mid, peak_gbs, b_link or peak_gbs)
    t_pred_ms = L * mdl["t_pred_us"] / 1000.0
    eqbw = {"alpha_measured": alpha, "b_gpu_gbs": peak_gbs, "b_link_gbs": b_link or peak_gbs,
            "b_link_kind": "page-locked host to HBM copy, measured" if b_link else "values in HBM",
            "eq_bandwidth_gbs": mdl["eq_bandwidth_gbs"], "t_pred_ms_per_step": t_pred_ms,
            "t_meas_ms_per_step": ms / K, "meas_over_pred": (ms / K) / t_pred_ms}

    thp1 = thp_counters()
    st_all = [lay.stats(check=False) for lay in layers]
    dev_err = [s["device_error"] for s in st_all if s["device_error"]]
    for lay in layers:
        lay.close()
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return None

    tokens_s = ws * w.batch * K / (ms / 1000.0)
    step_ms = ms / K
    hbm_per_step = hbm / K
    line = {
        "metric": METRIC, "value": tokens_s, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16+e5m2" if w.dtype == "fp8" else w.dtype,
        "data": "synthetic (seeded generator; Llama-3.1-8B attention shape)",
        "config": {**workload_config(w, L),
                   "parallelism": f"replicas x{ws} (batch sharded, no collective)",
                   "microbatches": M,
                   "layers_share_input_storage": share,
                   "host_values": ({"pinned": "one page-locked arena (shadowkv_host_alloc_kind, SKV_HOST_PINNED)",
                                    "huge": "one arena of transparent huge pages read through the host page tables "
                                            "(shadowkv_host_alloc_kind, SKV_HOST_HUGE)"}[args.host_mem]
                                   if w.v_place == "host" else None),
                   "l2": "inputs larger than L2 (landmarks of one layer exceed 129 MB)"},
        "hbm_gbs": hbm_per_step / (step_ms * 1e-3) / 1e9,
        "hbm_frac_of_8tbs": hbm_per_step / 8e12 / (step_ms * 1e-3),
        "hbm_bytes_per_step": hbm_per_step, "link_bytes_per_step": link / K,
        "link_gbs": (link / K) / (step_ms * 1e-3) / 1e9, "scratch_bytes_per_step": scratch / K,
        "alpha_mean": alpha,
        "roofline": {"bound": "hbm", "kernel": "k_score (landmark scoring)", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": score_traffic,
                     "algorithmic_bytes_per_launch": score_bytes, "avg_launch_us": score_us},
        "phase_ms_per_step": {ph: phase_ms[ph] / K for ph in skv.PHASES},
        "eq_bandwidth_check": eqbw,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches,
        "setup_s": setup_s,
        "host_thp_counters_delta": {k: thp1.get(k, 0) - thp0.get(k, 0) for k in thp1},
    }
    if dev_err:
        line["device_error"] = dev_err[0]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, seconds=12.0)
    if ws > 1:
        dist.destroy_process_group()
    return line


def workload_config(w: Workload, layers: int) -> dict:
    """The workload part of the JSON line's config, the same for both arms."""
    return {"workload": w.name, "layers": layers, "batch_per_gpu": w.batch, "seq_len": w.seq_len,
            "n_kv_heads": w.n_kv_heads, "n_q_heads": w.n_q_heads, "head_dim": w.head_dim,
            "rank": w.rank, "chunk": w.chunk, "n_select": w.n_select, "n_outlier": w.n_outlier,
            "local_window": w.local_window, "v_place": w.v_place, "drift": w.drift,
            "new_keys": w.new_keys, "dtype": w.dtype}


# ----------------------------------------------------------------------------- oracle arm
class OracleSample:
    """The float64 oracle's decode step on one (batch, KV head) unit of layer 0,
    on this host's cores.  Inputs of that unit come from the same seeded
    generator (CPU stream); the oracle's pre-filling of the unit is untimed."""

    def __init__(self, w: Workload, unit: int = 0, max_steps: int = 4096):
        from oracle import shadowkv_ref as ref
        from workload import make_A, make_B, make_decode_inputs, make_V
        self.ref, self.w = ref, w
        b, h = divmod(unit, w.n_kv_heads)
        one = w.with_(batch=b + 1)
        self.A = make_A(one, 0, "cpu")[b].double().numpy()
        self.B = make_B(one, 0, "cpu")[b, h].double().numpy()
        self.V = make_V(one.with_(n_kv_heads=h + 1), 0, "cpu")[b, h].double().numpy()
        q, kn, vn = make_decode_inputs(one, 0, min(max_steps, 256), "cpu")
        G = w.group
        self.q = q[:, b, h * G:(h + 1) * G].double().numpy()
        self.kn, self.vn = kn[:, b, h].double().numpy(), vn[:, b, h].double().numpy()
        t0 = time.perf_counter()
        self.st = ref.UnitDecodeState(ref.prefill_unit(self.A, self.B, self.V, w.chunk, w.n_outlier,
                                                       w.local_window, w.rope_base))
        self.prefill_s = time.perf_counter() - t0
        self.t = 0

    def timed_steps(self, budget_s: float, cap: int = 1 << 30):
        """Run unit-steps until ``budget_s`` of oracle time; returns (seconds per unit-step, n)."""
        w, ref = self.w, self.ref
        timed, n = 0.0, 0
        while n < cap and (n == 0 or timed < budget_s):
            t = self.t % self.q.shape[0]
            if self.st.steps >= self.q.shape[0]:
                self.st.pre.k_local = self.st.pre.k_local[: w.local_window]
                self.st.pre.v_local = self.st.pre.v_local[: w.local_window]
                self.st.steps = 0
            t1 = time.perf_counter()
            ref.decode_step_unit(self.st, self.q[t], self.kn[t], self.vn[t], self.A, self.B, self.V,
                                 w.n_select, w.chunk, w.rope_base)
            timed += time.perf_counter() - t1
            n += 1
            self.t += 1
        return timed / n, n


def cpu_baseline(w: Workload, seconds: float = 12.0) -> dict:
    o = OracleSample(w)
    per_unit, n = o.timed_steps(seconds)
    step_s = per_unit * w.units * w.layers
    return {"value": w.batch / step_s, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"{n} oracle decode steps of one (batch, KV head) unit of layer 0 ({per_unit * 1e3:.1f} ms "
                       f"each), scaled to {w.units} units x {w.layers} layers per decode step; the unit's "
                       f"oracle pre-filling ({o.prefill_s:.1f} s) untimed; numpy BLAS may use every host core")}


def run_reference(args, w: Workload, ws: int, rank: int):
    if rank != 0:
        return None
    K, W = args.steps, args.warmup
    budget = args.ref_budget if args.ref_budget > 0 else max(0.5, min(10.0, 120.0 / max(1, K + W)))
    o = OracleSample(w)
    for _ in range(W):
        o.timed_steps(budget / 4, cap=2)
    per = [o.timed_steps(budget)[0] for _ in range(K)]
    per_unit = statistics.mean(per)
    step_s = per_unit * w.units * w.layers
    v = w.batch / step_s
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": W, "ms_per_step": step_s * 1000.0, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
        "config": {**workload_config(w, w.layers), "parallelism": "oracle on the host cores (rank 0 only)"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": (f"each step: float64 oracle decode steps of one unit of layer 0 for about "
                                    f"{budget:.1f} s, scaled to {w.units} units x {w.layers} layers")},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    ws, rank, local = dist_env()
    w = workload_from(args)
    if args.impl == "reference":
        line = run_reference(args, w, ws, rank)
    else:
        line = run_ours(args, w, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
