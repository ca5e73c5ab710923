"""Decode-step benchmark of the ShadowKV sparse-attention path on GB300.

One step = one decode step of every layer (all rows of the hot path: landmark
scoring, top-K + index scan + append, key rebuild, value fetch, sparse
attention) for the whole batch.  Default workload: Llama-3.1-8B attention
shape at 128K context, batch 8, 32 layers, values in host memory.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
of the workload (independent batches, no collective on the data path) and the
timing is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
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
HBM_NOMINAL_GBS = 8000.0
EQBW_TOLERANCE = 0.25   # measured step time within +-25 % of the equivalent-bandwidth prediction
HUGE_SPLIT_LIMIT = 0.25  # more huge-page splits than this share of the arena's pages during setup: page-locked


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    # page-locked host values run slow for about a second after a fresh arena is filled on a box
    # (measured, the first run on a box: 702 tokens/s after 5 warm-up steps, 1029 after 100)
    ap.add_argument("--warmup", type=int, default=100)
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
    ap.add_argument("--ref-workers", type=int, default=0,
                    help="oracle worker processes of the reference arm and the CPU baseline (default: every "
                         "host core)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-hbm-sub", action="store_true",
                    help="skip the values-in-HBM sub-result of a host-values run")
    ap.add_argument("--microbatches", type=int, default=1,
                    help="split the batch into this many handles per layer, each on its own stream pair")
    ap.add_argument("--pipeline", action="store_true",
                    help="with --microbatches M >= 2: stagger the micro-batches, each one's scoring waits for "
                         "the previous one's selection, so one's value fetch overlaps the next one's scoring")
    ap.add_argument("--host-mem", default="pinned", choices=["pinned", "huge"],
                    help="host values: page-locked memory, or transparent huge pages read through the host "
                         "page tables (faster while the host kernel keeps the pages whole)")
    ap.add_argument("--single-stream", action="store_true",
                    help="run the value fetch on the main stream too (fetch, then rebuild)")
    return ap.parse_args(argv)


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
    keys = ("thp_split_pmd", "thp_split_page", "thp_fault_alloc", "pgmigrate_success", "thp_collapse_alloc")
    out = {}
    try:
        for line in open("/proc/vmstat"):
            k, _, v = line.partition(" ")
            if k in keys:
                out[k] = int(v)
    except OSError:
        pass
    return out


def huge_storm(splits: int, pages: float) -> bool:
    """A huge-page arena whose setup split more than HUGE_SPLIT_LIMIT of its pages: measured, the
    host kernel then keeps splitting, and the bench measures with page-locked values instead."""
    return splits > HUGE_SPLIT_LIMIT * pages


def mem_available_gb() -> float:
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) / 1e6
    except OSError:
        pass
    return 0.0


def device_bytes_estimate(w: Workload, per_layer_inputs: bool) -> float:
    """Device bytes a run of every layer holds: the library's state per layer (landmarks, chunk
    ids, logits and selection scratch, the attended key/value blocks) plus A, B and (values in
    HBM) V, per layer or once when the layers share their inputs."""
    es, es_l, es_v = elem_sizes(w)
    U, d, nc = w.units, w.head_dim, w.n_selectable
    rows = (w.n_outlier + w.n_select) * w.chunk + w.local_window + w.steps
    state = U * (nc * (d * es_l + 4 + 4 * w.group + 8) + rows * d * (es + es_v) + w.n_chunks * 4)
    inputs = w.batch * w.seq_len * w.rank * es + U * w.rank * d * es
    if w.v_place == "hbm":
        inputs += U * w.seq_len * d * es_v
    return w.layers * state + (w.layers if per_layer_inputs else 1) * inputs


def elem_sizes(w: Workload):
    """Bytes per element of (keys, factors, q, out), of the landmarks and of the values."""
    es = 4 if w.dtype == "f32" else 2
    es_lv = 1 if w.dtype == "fp8" else es
    return es, es_lv, es_lv


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
class Run:
    """Every layer of a workload prefilled on the GPU, with per-step decode inputs in HBM."""

    def __init__(self, args, w: Workload, dev, total_steps: int, ws: int):
        import torch

        import sparse_kv_cache_gb300 as skv
        from workload import make_A, make_B, make_decode_inputs, make_V, storage_dtype, value_dtype

        self.args, self.w, self.dev, self.ws = args, w, dev, ws
        self.skv, self.torch = skv, torch
        L = w.layers
        self.dt, self.vdt = storage_dtype(w), value_dtype(w)   # keys, factors, q, out / values
        es_v = elem_sizes(w)[2]
        v_bytes = w.batch * w.n_kv_heads * w.seq_len * w.head_dim * es_v
        share = args.share_storage == "yes"
        if args.share_storage == "auto":
            if w.v_place == "host":
                share = mem_available_gb() < 1.3 * L * v_bytes / 1e9 + 16
            else:
                share = device_bytes_estimate(w, per_layer_inputs=True) > 0.85 * torch.cuda.mem_get_info(dev)[0]
        self.share = share
        n_data = 1 if share else L
        M = self.M = max(1, args.microbatches)
        if w.batch % M:
            raise SystemExit(f"batch {w.batch} is not a multiple of --microbatches {M}")
        bm = self.bm = w.batch // M
        self.arena = None
        if w.v_place == "host":
            # one arena for every layer's values (large allocations keep GPU translations few)
            per = w.batch * w.n_kv_heads * w.seq_len * w.head_dim
            self.arena = skv.HostBuffer((n_data * per,), self.vdt, kind=args.host_mem)
        # one (main, side) stream pair per micro-batch; the value fetch (link-bound) goes first
        self.mains = [torch.cuda.Stream(dev) for _ in range(M)]
        self.sides = [torch.cuda.Stream(dev, priority=-10) for _ in range(M)]
        self.main = self.mains[0]
        data, layers = [], []
        t0 = time.time()
        for ell in range(n_data):
            A = make_A(w, ell, dev)
            B = make_B(w, ell, dev)
            Vd = make_V(w, ell, dev)
            if w.v_place == "host":
                # values stay in host memory; the GPU reads missed chunks in place over NVLink-C2C
                self.arena.fill_from(Vd, ell * Vd.numel())
                V = self.arena.slice(ell * Vd.numel(), Vd.shape)
                del Vd
            else:
                V = Vd
            data.append((A, B, V))
        fill_counters = thp_counters()
        # micro-batch m owns batch rows [m*bm, (m+1)*bm) of every tensor (all are batch-major)
        cfg = skv.make_config(w.with_(batch=bm), max_new_tokens=total_steps)
        for ell in range(L):
            A, B, V = data[ell % n_data]
            for m in range(M):
                rows = slice(m * bm, (m + 1) * bm)
                layers.append(skv.Layer(cfg, A[rows], B[rows], V[rows], stream=self.main))
        torch.cuda.synchronize()
        self.setup_s = time.time() - t0
        self.data, self.layers = data, layers
        self.thp_trace = {"after_fill": fill_counters, "after_prefill": thp_counters()}
        # per-layer decode inputs for every step, resident in HBM
        self.qs, self.kns, self.vns = [], [], []
        for ell in range(L):
            q, kn, vn = make_decode_inputs(w, ell, total_steps, dev)
            self.qs.append(q)
            self.kns.append(kn)
            self.vns.append(vn)
        self.out = [torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=self.dt, device=dev) for _ in range(L)]
        self.hq = [lay.handle for lay in layers]
        self.lib = skv.load()
        self.ms_ = [st.cuda_stream for st in self.mains]
        self.ss_ = [None if args.single_stream else st.cuda_stream for st in self.sides]
        self.pipe = args.pipeline and M >= 2
        self.sel_ev = []
        if self.pipe:
            # micro-batch m of layer ell scores after micro-batch m-1 of that layer has selected
            # (micro-batch 0 after the last one of the layer before, across steps too)
            for ell in range(L):
                for m in range(M):
                    e = torch.cuda.Event()
                    layers[ell * M + m].set_select_event(e)
                    self.sel_ev.append(e)
        self.s_idx = 0

    def stagger(self, ell: int, m: int):
        if self.pipe:
            prev = ell * self.M + m - 1
            self.mains[m].wait_event(self.sel_ev[prev if prev >= 0 else self.w.layers * self.M - 1])

    def step(self):
        s, M, bm, lib = self.s_idx, self.M, self.bm, self.lib
        # layer order is kept within each micro-batch's stream; the micro-batches run side by side
        for ell in range(self.w.layers):
            for m in range(M):
                self.stagger(ell, m)
                rows = slice(m * bm, (m + 1) * bm)
                rc = lib.shadowkv_decode_step(self.hq[ell * M + m], self.qs[ell][s][rows].data_ptr(),
                                              self.kns[ell][s][rows].data_ptr(), self.vns[ell][s][rows].data_ptr(),
                                              self.out[ell][rows].data_ptr(), None, self.ms_[m], self.ss_[m])
                if rc:
                    raise self.skv.ShadowKVError(rc, "decode_step")
        self.s_idx += 1

    def fork(self, ev):
        for st in self.mains[1:]:
            st.wait_event(ev)

    def join(self):
        for st in self.mains[1:]:
            ev = self.torch.cuda.Event()
            ev.record(st)
            self.main.wait_event(ev)

    def barrier(self):
        self.torch.cuda.synchronize()
        if self.ws > 1:
            import torch.distributed as dist
            dist.barrier()
        self.torch.cuda.synchronize()

    def timed(self, K: int) -> float:
        """K steps between two events on the main stream (forked to every micro-batch); ms."""
        torch = self.torch
        self.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.main)
        self.fork(e0)
        for _ in range(K):
            self.step()
        self.join()
        e1.record(self.main)
        self.barrier()
        return e0.elapsed_time(e1)

    def reset_stats(self):
        for lay in self.layers:
            lay.reset_stats()

    def stats(self, check: bool = True):
        return [lay.stats(check=check) for lay in self.layers]

    def e2e(self, K: int) -> dict:
        """K steps end to end through the public call with host buffers.  Every step copies its
        inputs (q, k_new, v_new of every layer, packed in one page-locked buffer) to the device in
        one copy and reads every layer's output back in one copy, both on a copy stream; the
        device buffers are double-buffered so the next step's inputs arrive while this step
        computes.  The timed region holds all K steps' copies."""
        torch, w, L, M, bm = self.torch, self.w, self.w.layers, self.M, self.bm
        es = elem_sizes(w)[0]
        qs, kns, vns, dt, dev = self.qs, self.kns, self.vns, self.dt, self.dev
        s0 = self.s_idx
        nq, nk, nv = qs[0][0].numel(), kns[0][0].numel(), vns[0][0].numel()
        per_layer = nq + nk + nv
        hin = torch.empty((K, L, per_layer), dtype=dt, pin_memory=True)
        for k in range(K):
            for ell in range(L):
                hin[k, ell, :nq].copy_(qs[ell][s0 + k].reshape(-1))
                hin[k, ell, nq:nq + nk].copy_(kns[ell][s0 + k].reshape(-1))
                hin[k, ell, nq + nk:].copy_(vns[ell][s0 + k].reshape(-1))
        oshape = tuple(self.out[0].shape)
        din = [torch.empty((L, per_layer), dtype=dt, device=dev) for _ in range(2)]
        dout = [torch.empty((L,) + oshape, dtype=dt, device=dev) for _ in range(2)]
        hout = torch.empty((K, L) + oshape, dtype=dt, pin_memory=True)
        cs = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(K)]
        ev_done = [torch.cuda.Event() for _ in range(K)]     # step k's kernels finished (main)
        ev_read = [torch.cuda.Event() for _ in range(K)]     # step k's outputs copied back (cs)
        self.barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(self.main)
        self.fork(f0)
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
                self.mains[m].wait_event(ev_in[k])
                if k >= 2:
                    self.mains[m].wait_event(ev_read[k - 2])  # dout[k % 2] was read back
            for ell in range(L):
                qv = b_in[ell, :nq].view(qs[ell][0].shape)
                kv = b_in[ell, nq:nq + nk].view(kns[ell][0].shape)
                vv = b_in[ell, nq + nk:].view(vns[ell][0].shape)
                for m in range(M):
                    self.stagger(ell, m)
                    rows = slice(m * bm, (m + 1) * bm)
                    self.layers[ell * M + m].decode_step(qv[rows], kv[rows], vv[rows], b_out[ell][rows], None,
                                                         main=self.mains[m],
                                                         side=None if self.args.single_stream else self.sides[m])
            self.join()
            ev_done[k].record(self.main)
            cs.wait_event(ev_done[k])
            with torch.cuda.stream(cs):
                hout[k].copy_(b_out, non_blocking=True)
            ev_read[k].record(cs)
        self.main.wait_event(ev_read[K - 1])
        self.join()
        f1.record(self.main)
        self.barrier()
        ms_e2e = max_over_ranks(f0.elapsed_time(f1), self.ws, dev)
        self.s_idx += K
        return {"value": self.ws * w.batch * K / (ms_e2e / 1000.0), "unit": UNIT,
                "h2d_bytes_per_step": L * per_layer * es, "d2h_bytes_per_step": L * self.out[0].numel() * es}

    def link_peaks(self, misses_per_layer: int) -> dict:
        """The host link measured live: a sequential page-locked host -> HBM copy of 256 MB, and
        the decode step's fetch kernel reading random chunks (address order, one layer's worth of
        misses) over the whole value arena, both with warm translations (the same chunks each
        time) and with fresh chunks every time, as successive layers' fetches read them."""
        torch, dev, w = self.torch, self.dev, self.w
        n = 256 << 20
        src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        src.fill_(1)
        dbuf = torch.empty(n, dtype=torch.uint8, device=dev)
        dbuf.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(3):
            dbuf.copy_(src, non_blocking=True)
        c1.record()
        torch.cuda.synchronize()
        seq = 3 * n / (c0.elapsed_time(c1) * 1e-3) / 1e9
        del dbuf, src
        chunk = w.chunk * w.head_dim * elem_sizes(w)[2]
        m = max(1, misses_per_layer)
        s = torch.cuda.current_stream()
        warm = self.skv.fetch_probe(self.arena.data_ptr(), self.arena.nbytes, m, chunk, seed=11, reps=3, stream=s)
        cold = self.skv.fetch_probe(self.arena.data_ptr(), self.arena.nbytes, m, chunk, seed=12, reps=3,
                                    fresh=True, stream=s)
        return {"seq_copy_gbs": seq, "random_chunk_warm_gbs": warm, "random_chunk_fresh_gbs": cold,
                "chunk_bytes": chunk, "chunks": m,
                "how": ("sequential: 3 x 256 MB page-locked host -> HBM copies (CUDA events); random: "
                        f"{m} distinct random {chunk}-byte chunks over the whole value arena read by the decode "
                        "step's fetch kernel in address order, best of 3, the same chunks each time (warm) or "
                        "new ones each time (fresh)")}

    def close(self):
        for lay in self.layers:
            lay.close()
        self.layers = []
        self.data = []
        if self.arena is not None:
            self.arena.free()
            self.arena = None


def kernel_rooflines(w: Workload, M: int, st2: list, phase_ms: dict, phase_n: dict, t_mid: int,
                     peak_hbm: float, link_peak: float | None) -> list:
    """Per-kernel achieved rates in the profiled pass: algorithmic bytes per launch (the decode
    step's byte model, split by kernel) over the average event-timed launch."""
    es, es_l, es_v = elem_sizes(w)
    U = w.units // M
    d, C, r, G = w.head_dim, w.chunk, w.rank, w.group
    n_launch = max(1, phase_n["score"])
    misses = sum(s["misses"] for s in st2) / n_launch               # missed chunks per launch
    rows_attn = w.n_outlier * C + w.n_select * C + w.local_window + t_mid + 1
    host = w.v_place == "host"
    spec = [
        ("score", "k_score_tc (landmark scoring)", "hbm", U * (w.n_selectable * es_l + G * es) * d),
        ("select", "k_select_decode (softmax, group max, top-K, index scan, append)", "latency",
         U * w.n_selectable * G * 4),
        ("rebuild", "k_rebuild_tc (gather A rows, A.B, RoPE)", "hbm", misses * C * es * (r + d) + U * r * d * es),
        ("fetch", "k_gather2 (value fetch, two chunks per warp)", "link" if host else "hbm", misses * C * d * es_v * (1 if host else 2)),
        ("attn", "k_attn_tc + k_attn_merge (split-K attention)", "hbm",
         U * (rows_attn * d * (es + es_v) + 2 * G * d * es)),
    ]
    rows = []
    for ph, name, bound, nbytes in spec:
        if ph == "fetch" and phase_n[ph] == 0:
            continue   # values in HBM read in place by attention: no fetch kernel
        n = max(1, phase_n[ph])
        us = 1000.0 * phase_ms[ph] / n
        gbs = nbytes / (us * 1e-6) / 1e9 if us > 0 else 0.0
        peak = link_peak if (bound == "link" and link_peak) else peak_hbm
        rows.append({"phase": ph, "kernel": name, "bound": bound, "bytes_per_launch": nbytes,
                     "bytes_kind": "scratch logits read" if ph == "select" else "algorithmic",
                     "avg_launch_us": us, "launches": phase_n[ph], "achieved_gbs": gbs, "peak_gbs": peak,
                     "frac": gbs / peak if peak else None})
    return rows


def run_ours(args, w: Workload, ws: int, rank: int, local: int):
    import torch
    import torch.distributed as dist

    import sparse_kv_cache_gb300 as skv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    K, W = args.steps, args.warmup
    passes = 3
    total_steps = W + passes * K
    w = w.with_(seed=replica_seed(w.seed, rank), steps=total_steps)
    L = w.layers
    peak_hbm, peak_kind = measured_peaks()
    thp0 = thp_counters()

    R = Run(args, w, dev, total_steps, ws)
    M = R.M
    for _ in range(W):
        R.step()
    torch.cuda.synchronize()
    repair, fallback = None, None
    if R.arena is not None and R.arena.kind == "huge":
        # huge pages split during the warm-up steps are put back together before timing
        t_r = time.time()
        rc = R.arena.repair()
        repair = {"status": rc, "seconds": time.time() - t_r}
        splits = thp_counters().get("thp_split_pmd", 0) - thp0.get("thp_split_pmd", 0)
        pages = R.arena.nbytes / (512 << 20)
        if huge_storm(splits, pages):
            # the host kernel kept splitting the arena's huge pages while it was filled and the
            # layers pre-filled (measured once: 86 of 128): measure with page-locked values instead
            import copy
            fallback = {"from": "huge", "to": "pinned", "splits_during_setup": splits,
                        "huge_pages": pages, "limit_fraction": HUGE_SPLIT_LIMIT}
            R.close()
            del R
            args = copy.copy(args)
            args.host_mem = "pinned"
            R = Run(args, w, dev, total_steps, ws)
            for _ in range(W):
                R.step()
            torch.cuda.synchronize()
    R.reset_stats()
    R.thp_trace["after_warmup_and_repair"] = thp_counters()

    # ---- pass 1: device-resident inputs (the headline value)
    clocks = ClockSampler(local)
    clocks.start()
    ms = max_over_ranks(R.timed(K), ws, dev)
    clk = clocks.stop()
    R.thp_trace["after_timed_pass"] = thp_counters()
    st = R.stats()
    hbm = sum(s["hbm_bytes"] for s in st)
    link = sum(s["link_bytes"] for s in st)
    scratch = sum(s["scratch_bytes"] for s in st)
    alpha = statistics.mean(s["alpha_mean"] for s in st)
    launches = int(sum(s["kernel_launches"] for s in st))   # the library's own count per decode step

    # ---- pass 2: the same steps with per-phase CUDA events; its own total is kept beside the
    # headline's (events between kernels cost the programmatic-launch overlap)
    R.reset_stats()
    for lay in R.layers:
        lay.set_profiling(True)
    t_prof = R.s_idx
    ms_prof = R.timed(K)
    st2 = R.stats()
    for lay in R.layers:
        lay.set_profiling(False)
    phase_ms = {ph: sum(s["phase_ms"][ph] for s in st2) for ph in skv.PHASES}
    phase_n = {ph: sum(s["phase_launches"][ph] for s in st2) for ph in skv.PHASES}

    R.thp_trace["after_profiled_pass"] = thp_counters()
    # ---- pass 3: end to end through the public call with host buffers
    e2e = None if args.no_e2e else R.e2e(K)
    R.thp_trace["after_e2e_pass"] = thp_counters()

    misses_layer = int(round(sum(s["misses"] for s in st2) / max(1, K) / L))
    links = R.link_peaks(misses_layer) if R.arena is not None else None
    thp1 = thp_counters()
    dev_err = [s["device_error"] for s in R.stats(check=False) if s["device_error"]]
    share, setup_s = R.share, R.setup_s
    thp_trace = {k: {c: v.get(c, 0) - thp0.get(c, 0) for c in ("thp_split_pmd", "pgmigrate_success", "thp_collapse_alloc")}
                 for k, v in R.thp_trace.items()}
    R.close()
    del R

    step_ms = ms / K
    hbm_step, link_step = hbm / K, link / K
    link_peak = links["seq_copy_gbs"] if links else None
    t_mid = W + K + K // 2
    kernels = kernel_rooflines(w, M, st2, phase_ms, phase_n, t_prof + K // 2, peak_hbm, link_peak)
    by = {k["phase"]: k for k in kernels}
    # the step against its binding term: the larger of its HBM and host-link times
    t_hbm = hbm_step / (peak_hbm * 1e9) * 1e3
    t_link = link_step / (link_peak * 1e9) * 1e3 if link_peak else 0.0
    binding = "link" if t_link > t_hbm else "hbm"
    dom = by["fetch"] if binding == "link" and "fetch" in by else max(
        (k for k in kernels if k["bound"] == "hbm"), key=lambda k: k["avg_launch_us"] * k["launches"])
    traffic = score_traffic_per_launch(w.with_(batch=w.batch // M)) if dom["phase"] == "score" else None
    roofline = {
        "bound": dom["bound"], "kernel": dom["kernel"], "achieved": dom["achieved_gbs"], "peak": dom["peak_gbs"],
        "unit": "GB/s", "frac": dom["frac"],
        "peak_kind": ("host link: sequential page-locked copy, measured live" if dom["bound"] == "link"
                      else f"HBM copy, {peak_kind} (MEASURED_PEAKS.json)"),
        "traffic": traffic, "algorithmic_bytes_per_launch": dom["bytes_per_launch"],
        "avg_launch_us": dom["avg_launch_us"],
        "step": {"ms": step_ms, "hbm_bytes": hbm_step, "link_bytes": link_step,
                 "t_hbm_ms": t_hbm, "t_link_ms": t_link, "binding": binding,
                 "frac_of_binding": max(t_hbm, t_link) / step_ms,
                 "hbm_frac_of_measured": t_hbm / step_ms,
                 "hbm_frac_of_8tbs": hbm_step / (HBM_NOMINAL_GBS * 1e9) / (step_ms * 1e-3)},
        "kernels": kernels,
    }
    if links and dom["bound"] == "link":
        roofline["frac_of_random_chunk_warm"] = dom["achieved_gbs"] / links["random_chunk_warm_gbs"]
        roofline["frac_of_random_chunk_fresh"] = dom["achieved_gbs"] / links["random_chunk_fresh_gbs"]

    # the pages' equivalent-bandwidth model with the measured hit rate and bandwidths: predicted step time
    cfg_m = skv.make_config(w, max_new_tokens=total_steps)
    mdl = skv.model(cfg_m, max(0.0, min(1.0, alpha)), t_mid, peak_hbm, link_peak or peak_hbm)
    t_pred_ms = L * mdl["t_pred_us"] / 1000.0
    ratio = step_ms / t_pred_ms
    eqbw = {"alpha_measured": alpha, "b_gpu_gbs": peak_hbm, "b_link_gbs": link_peak or peak_hbm,
            "b_link_kind": "page-locked host to HBM copy, measured live" if link_peak else "values in HBM",
            "eq_bandwidth_gbs": mdl["eq_bandwidth_gbs"], "t_pred_ms_per_step": t_pred_ms,
            "t_meas_ms_per_step": step_ms, "meas_over_pred": ratio, "tolerance": EQBW_TOLERANCE,
            "within_tolerance": abs(ratio - 1.0) <= EQBW_TOLERANCE}

    # values-in-HBM sub-result of a host-values run: the same workload and steps, values in HBM
    sub = None
    if w.v_place == "host" and not args.no_hbm_sub:
        w2 = w.with_(v_place="hbm", steps=W + K)
        R2 = Run(args, w2, dev, W + K, ws)
        for _ in range(W):
            R2.step()
        R2.reset_stats()
        ms2 = max_over_ranks(R2.timed(K), ws, dev)
        hbm2 = sum(s["hbm_bytes"] for s in R2.stats()) / K
        R2.close()
        del R2
        sub = {"v_place": "hbm", "value": ws * w.batch * K / (ms2 / 1000.0), "unit": UNIT, "ms_per_step": ms2 / K,
               "hbm_bytes_per_step": hbm2,
               "hbm_frac_of_measured": hbm2 / (peak_hbm * 1e9) / (ms2 / K * 1e-3),
               "hbm_frac_of_8tbs": hbm2 / (HBM_NOMINAL_GBS * 1e9) / (ms2 / K * 1e-3),
               "how": "the same workload and steps with the values in HBM (fresh handles), timed pass only"}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return None

    tokens_s = ws * w.batch * K / (ms / 1000.0)
    two = not args.single_stream
    crit = (phase_ms["score"] + phase_ms["select"] + phase_ms["attn"] +
            (max(phase_ms["rebuild"], phase_ms["fetch"]) if two else phase_ms["rebuild"] + phase_ms["fetch"]))
    line = {
        "metric": METRIC, "value": tokens_s, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16+e5m2" if w.dtype == "fp8" else w.dtype,
        "data": "synthetic (seeded generator; Llama-3.1-8B attention shape)",
        "config": line_config(args, w, L, ws),
        "run": {"microbatches": M, "pipelined": args.pipeline and M >= 2, "single_stream": args.single_stream,
                "layers_share_input_storage": share,
                "host_values": ({"pinned": "one page-locked arena (shadowkv_host_alloc_kind, SKV_HOST_PINNED)",
                                 "huge": "one arena of transparent huge pages read through the host page tables "
                                         "(shadowkv_host_alloc_kind, SKV_HOST_HUGE)"}[args.host_mem]
                                if w.v_place == "host" else None)},
        "hbm_gbs": hbm_step / (step_ms * 1e-3) / 1e9,
        "hbm_frac_of_8tbs": hbm_step / (HBM_NOMINAL_GBS * 1e9) / (step_ms * 1e-3),
        "hbm_frac_of_measured": hbm_step / (peak_hbm * 1e9) / (step_ms * 1e-3),
        "hbm_bytes_per_step": hbm_step, "link_bytes_per_step": link_step,
        "link_gbs": link_step / (step_ms * 1e-3) / 1e9, "scratch_bytes_per_step": scratch / K,
        "link_peaks": links,
        "alpha_mean": alpha,
        "roofline": roofline,
        "phase_ms_per_step": {ph: phase_ms[ph] / K for ph in skv.PHASES},
        "phase_split": {"profiled_pass_ms_per_step": ms_prof / K, "critical_path_ms_per_step": crit / K,
                        "timed_pass_ms_per_step": step_ms,
                        "note": ("the split comes from a second pass with events between kernels, which cost the "
                                 "programmatic-launch overlap; both totals stand beside the timed pass's")},
        "eq_bandwidth_check": eqbw,
        "v_place_hbm": sub,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches,
        "setup_s": setup_s,
        "host_thp_counters_delta": {k: thp1.get(k, 0) - thp0.get(k, 0) for k in thp1},
        "host_thp_trace": thp_trace,
        "host_repair_after_warmup": repair,
        "host_mem_fallback": fallback,
    }
    if dev_err:
        line["device_error"] = dev_err[0]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, workers=args.ref_workers)
    if ws > 1:
        dist.destroy_process_group()
    return line


def workload_config(w: Workload, layers: int) -> dict:
    """The workload part of the JSON line's config."""
    return {"workload": w.name, "layers": layers, "batch_per_gpu": w.batch, "seq_len": w.seq_len,
            "n_kv_heads": w.n_kv_heads, "n_q_heads": w.n_q_heads, "head_dim": w.head_dim,
            "rank": w.rank, "chunk": w.chunk, "n_select": w.n_select, "n_outlier": w.n_outlier,
            "local_window": w.local_window, "v_place": w.v_place, "drift": w.drift,
            "new_keys": w.new_keys, "dtype": w.dtype}


def line_config(args, w: Workload, layers: int, ws: int) -> dict:
    """The JSON line's config: the same dict from both arms for the same command line."""
    return {**workload_config(w, layers),
            "parallelism": f"replicas x{ws} (batch sharded, no collective)",
            "l2": "inputs larger than L2 (the landmarks of one layer exceed 129 MB)"}


# ----------------------------------------------------------------------------- oracle arm
class OracleSample:
    """The float64 oracle's decode step on one (batch, KV head) unit of layer 0, on this host's
    cores.  Inputs of that unit come from the same seeded generator (CPU stream); the oracle's
    pre-filling of the unit is untimed."""

    def __init__(self, w: Workload, unit: int = 0, max_steps: int = 4096):
        from oracle import shadowkv_ref as ref
        from workload import make_A, make_B, make_decode_inputs, make_V
        self.ref, self.w = ref, w
        b, h = divmod(unit % w.units, w.n_kv_heads)
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

    def run_steps(self, n: int):
        w, ref = self.w, self.ref
        for _ in range(n):
            t = self.t % self.q.shape[0]
            if self.st.steps >= self.q.shape[0]:
                self.st.pre.k_local = self.st.pre.k_local[: w.local_window]
                self.st.pre.v_local = self.st.pre.v_local[: w.local_window]
                self.st.steps = 0
            ref.decode_step_unit(self.st, self.q[t], self.kn[t], self.vn[t], self.A, self.B, self.V,
                                 w.n_select, w.chunk, w.rope_base)
            self.t += 1


def _oracle_worker(w: Workload, unit: int, conn):
    """One oracle process: pre-fills one (batch, KV head) unit of layer 0 (untimed), then on
    each request runs n decode steps of it and answers with the seconds they took."""
    try:
        o = OracleSample(w, unit)
        conn.send(("ready", o.prefill_s))
        while True:
            msg = conn.recv()
            if msg is None:
                break
            t0 = time.perf_counter()
            o.run_steps(int(msg))
            conn.send(("done", time.perf_counter() - t0))
    except Exception as e:  # reported to the parent
        conn.send(("error", repr(e)))
    finally:
        conn.close()


BLAS_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


class OraclePool:
    """P oracle processes (spawned, one BLAS thread each), each on its own unit of layer 0."""

    def __init__(self, w: Workload, workers: int):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in BLAS_ENV}
        for k in BLAS_ENV:
            os.environ[k] = "1"
        self.procs, self.conns = [], []
        try:
            for i in range(workers):
                a, b = ctx.Pipe()
                p = ctx.Process(target=_oracle_worker, args=(w, i, b), daemon=True)
                p.start()
                self.procs.append(p)
                self.conns.append(a)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.prefill_s = []
        for c in self.conns:
            tag, v = c.recv()
            if tag != "ready":
                self.close()
                raise RuntimeError(f"oracle worker failed: {v}")
            self.prefill_s.append(v)

    def run(self, n: int) -> float:
        """Every worker runs n unit-steps at once; returns the wall seconds until the last is done."""
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(n)
        for c in self.conns:
            tag, v = c.recv()
            if tag != "done":
                raise RuntimeError(f"oracle worker failed: {v}")
        return time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except (OSError, BrokenPipeError):
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()


def cpu_baseline(w: Workload, workers: int = 0, budget_s: float = 3.0) -> dict:
    """The oracle as it stands on the host cores, single-threaded and with every core (one
    process per core, each on its own unit, one BLAS thread each), median of 3 timings each,
    scaled from unit-steps to decode steps of the whole workload (units x layers)."""
    P = workers or os.cpu_count() or 1
    one = OraclePool(w, 1)
    try:
        n1 = max(1, int(budget_s / max(1e-4, one.run(1))))
        singles = [one.run(n1) / n1 for _ in range(3)]
        pre1 = max(one.prefill_s)
    finally:
        one.close()
    pool = OraclePool(w, P)
    try:
        per = max(1, int(budget_s / max(1e-4, pool.run(1))))
        walls = [pool.run(per) for _ in range(3)]
    finally:
        pool.close()
    unit_steps = w.units * w.layers
    s1 = statistics.median(singles)                 # seconds per unit-step, one core
    sP = statistics.median(walls) / (per * P)       # seconds per unit-step, all cores
    return {"value": w.batch / (sP * unit_steps), "unit": UNIT, "cores": P, "kind": "oracle",
            "single_thread_value": w.batch / (s1 * unit_steps),
            "nproc": os.cpu_count(), "blas_threads_per_process": 1, "median_of": 3,
            "sample": (f"all cores: {P} spawned processes, each on its own (batch, KV head) unit of layer 0, "
                       f"{per} float64 oracle decode steps each per timing ({statistics.median(walls):.2f} s "
                       f"wall); one core: {n1} steps per timing ({s1 * 1e3:.1f} ms each); median of 3 timings "
                       f"each, scaled to {w.units} units x {w.layers} layers per decode step; the units' oracle "
                       f"pre-filling ({pre1:.1f} s each) untimed")}


def run_reference(args, w: Workload, ws: int, rank: int):
    """The oracle arm: each timed step runs float64 oracle decode steps on P units of layer 0 at
    once (P worker processes, one per host core); the line's value scales that measured step to
    the whole workload's decode step (units x layers unit-steps)."""
    if rank != 0:
        return None
    K, W = args.steps, args.warmup
    P = args.ref_workers or os.cpu_count() or 1
    pool = OraclePool(w, P)
    try:
        one = pool.run(1)
        target = args.ref_budget if args.ref_budget > 0 else max(0.2, min(5.0, 100.0 / max(1, K + W)))
        per = max(1, int(target / max(1e-4, one)))
        for _ in range(W):
            pool.run(per)
        walls = [pool.run(per) for _ in range(K)]
    finally:
        pool.close()
    step_s = statistics.mean(walls)                     # measured: `per` unit-steps on each of P units
    unit_steps = w.units * w.layers
    full_step_s = step_s / (per * P) * unit_steps       # the whole workload's decode step, scaled
    v = w.batch / full_step_s
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": W, "ms_per_step": step_s * 1000.0, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
        "config": line_config(args, w, w.layers, ws),
        "ms_per_step_kind": (f"measured: one timed step = {per} oracle decode steps on each of {P} units of "
                             f"layer 0 at once ({P} processes); value = batch / (that time x {unit_steps} / "
                             f"({per} x {P})), the whole workload's step scaled from the measured one"),
        "extrapolated_ms_per_full_step": full_step_s * 1000.0,
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": P, "kind": "oracle",
                         "sample": (f"each step: {per} float64 oracle decode steps on each of {P} units of "
                                    f"layer 0 in {P} spawned processes (one BLAS thread each), scaled to "
                                    f"{w.units} units x {w.layers} layers")},
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
