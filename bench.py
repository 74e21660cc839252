"""Benchmark of the predictive sparse-KV decode step on one GB300.

A step is one dd_decode_step over all L layers of a workload: scoring, top-k,
gather from the pinned host KV store and attention for every layer, on two
streams.  The default workload is the largest one that fits one GPU and its
host as stated: the high-concurrency GQA shape (32 layers cycling 4 distinct
layer slots, batch 32, 32 query / 8 KV heads x 128, context 131072, top-k
2048 per KV head, no window, bf16; 32 GiB of keys in HBM, 64 GiB of host K/V).
The 13B-shaped 64K workload would need 160 GiB of page-locked host memory for
its 8 layer slots, more than a 199 GiB host can lock beside everything else.

Prints one JSON line: layer-steps/s (device time, inputs resident; the median
of several back-to-back regions of K steps, with their min and max), the same
through the public API with host copies (e2e), the scoring kernel's HBM
roofline, the gather's host-link bandwidth against a pinned-copy probe taken in
the same process, the hidden fraction of the gather (event-free overlapped and
serial regions, interleaved), the recall of the prefetched rows, the step rate
as CUDA-graph replays, and the fp64 oracle timed on the host cores as the CPU
baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--repeats R]
                  [--impl ours|reference] [--workload NAME]
                  [--schedule auto|overlap|late|pipeline|serial|guarded]
                  [--landmarks C] [--fused-topk] [--correct-misses]
                  [--gather-mode 0|1] [--host-alloc pinned|huge|auto|torch] [--profile-case]

The host store defaults to driver-allocated page-locked memory.  The schedule
and the gather variant default to auto: overlap, serial, pipeline or guarded,
each with the small or wide bulk-copy gather or the load/store one, whichever
a short calibration after the warm-up measures fastest on this host and
workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "sparse-decode layer-steps/s; scoring HBM GB/s; gather host-link GB/s"
UNIT = "layer-steps/s"
FALLBACK_HBM_GBS = 6800.0
# DRAM read + write bytes of one scoring launch, from ncu captures of the
# current kernel (profiles/), scaled by units to the full layer.  GQA-128K: a
# batch-16 capture of the tensor-core form (128 units: 4.2954 GB read,
# 0.2204 GB of logits written, mean of two launches) doubled for the 256 units
# of the layer.  Keyed by (workload, top-k fused into the scoring kernel);
# absent where no capture of the current kernel exists.
SCORE_TRAFFIC_BYTES = {("c5-gqa-128k", False): 2 * (4295449856 + 220422528)}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=synth.C5.name, choices=list(synth.WORKLOADS))
    p.add_argument("--repeats", type=int, default=5,
                   help="back-to-back timed regions of --steps steps; value is the median")
    p.add_argument("--profile-case", action="store_true",
                   help="small case for ncu captures: batch --profile-batch, 2 layers, 1 slot")
    p.add_argument("--profile-batch", type=int, default=2,
                   help="batch of the --profile-case workload")
    p.add_argument("--gather-mode", type=int, default=None, choices=[0, 1],
                   help="0: bulk-copy gather, 1: load/store gather (default: chosen with the "
                        "schedule by the calibration; 0, or 1 with --landmarks, when the "
                        "schedule is given)")
    p.add_argument("--host-alloc", default="pinned", choices=["pinned", "huge", "auto", "torch"],
                   help="host KV store: dd_host_alloc_pinned (driver-allocated page-locked "
                        "memory, exact size; stable: the default), dd_host_alloc (locked "
                        "transparent huge pages: faster gathers while the host leaves them "
                        "alone, collapses when it splits and moves them), auto (the huge-page "
                        "store if its gathers reach steady state within --settle-seconds, else "
                        "the driver-allocated one; it can still collapse later), or torch "
                        "pinned memory")
    p.add_argument("--host-layout", default="interleaved", choices=["interleaved", "separate"],
                   help="host store layout: one store with each position's K row followed by "
                        "its V row (a position's two rows share a page: fewer translations), "
                        "or separate K and V stores")
    p.add_argument("--fill", default="auto", choices=["auto", "device", "cpu"],
                   help="how the host store is written: device-to-host copies of the "
                        "generated data (as a KV offload writes it), or CPU writes (auto)")
    p.add_argument("--copy-priority", default="high", choices=["high", "low"],
                   help="priority of the copy stream relative to the compute stream")
    p.add_argument("--slots", type=int, default=0,
                   help="override the number of distinct layer slots (memory-limited runs)")
    p.add_argument("--schedule", default="auto",
                   choices=["auto", "overlap", "late", "pipeline", "serial", "guarded"],
                   help="overlap: gather l+1 beside attention l; late: gather l+1 after "
                        "attention l; pipeline: gather and attention of each layer on the "
                        "copy stream; serial: every phase in order on one stream; guarded: "
                        "overlap, but each scoring waits for the previous layer's gather; "
                        "auto: overlap, serial, pipeline or guarded, whichever a short "
                        "calibration after the "
                        "warm-up measures fastest (scoring and the host gather slow each other "
                        "when they run together, by an amount that varies between hosts and "
                        "workloads)")
    p.add_argument("--correct-misses", action="store_true",
                   help="correct prediction misses in every timed layer (DD_STEP_CORRECT_MISSES)")
    p.add_argument("--landmarks", type=int, default=0, metavar="C",
                   help="select whole chunks of C rows by their mean-key landmarks "
                        "(DD_STEP_LANDMARKS) instead of scoring every key; 0: off")
    p.add_argument("--fused-topk", action="store_true",
                   help="steps 1-2 as one kernel whose last CTA per unit selects its rows "
                        "(DD_STEP_FUSED_TOPK) instead of scoring and top-k kernels")
    p.add_argument("--late-gather", type=int, default=0,
                   help="1: start each layer's gather after the previous attention")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="CPU work budget of the oracle baseline")
    p.add_argument("--settle-seconds", type=float, default=45.0,
                   help="longest wait for the host link to reach steady state before measuring")
    return p.parse_args()


# Gather variants the calibration tries: (tag, mode, geometry).  The small
# bulk-copy geometry fits beside the scoring kernel; the wide one keeps 5x the
# rows in flight, which pays on stores of small pages (translation latency);
# the half one keeps half the small one's rows in flight on half the SMs: on a
# store whose gather is bound by address translation, rows in flight beyond
# what the translations admit only wait, and they hold memory-system slots the
# scoring beside them needs; the load/store gather (eight warps per SM) takes
# no shared memory.  (Gathers on a quarter or 40 % of the SMs with 192 KiB of
# shared memory each, so that no scoring CTA shares their SMs, were 20-45 %
# slower per GQA-128K step than the small geometry and are not tried.)
GATHER_VARIANTS = (("bulk_copy_small", 0, (100, 4096, 3)),
                   ("bulk_copy_wide", 0, (200, 8192, 4)),
                   ("bulk_copy_half", 0, (50, 4096, 3)),
                   ("load_store", 1, (100, 256)))


def set_gather_variant(dd, mode, geom):
    if mode == 0:
        dd.set_gather_geometry(*geom)
    else:
        dd.set_gather_lsu_geometry(*geom)


def resolve_defaults(args):
    # The gather kernel is part of the automatic choice when the schedule is:
    # calibration then tries both (bulk copy and load/store).
    args.gather_auto = args.gather_mode is None and args.schedule == "auto"
    if args.gather_mode is None:
        args.gather_mode = 1 if args.landmarks else 0
    return args


def workload(args):
    w = synth.WORKLOADS[args.workload]
    if args.profile_case:
        w = w.scaled(batch=args.profile_batch, n_layers=2, n_slots=1)
    if args.slots:
        w = w.scaled(n_slots=args.slots)
    return w


# --------------------------------------------------------------- distributed

def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(layers_per_rank_step: int, steps: int, seconds_per_rank: float,
                   world: int) -> float:
    """Whole-job layer-steps/s: every rank runs its own replica (independent
    requests), so the job processes world x layers x steps layer-steps in the
    slowest rank's time (the caller passes the max over ranks)."""
    return world * layers_per_rank_step * steps / seconds_per_rank


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def anon_huge_bytes():
    """Bytes of this process's memory backed by transparent huge pages."""
    try:
        for line in open("/proc/self/smaps_rollup"):
            if line.startswith("AnonHugePages:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


VM_EVENTS = ("thp_split_pmd", "thp_split_page", "pgmigrate_success", "compact_migrate_scanned",
             "compact_isolated")


def vm_events():
    """Host memory-management event counters (/proc/vmstat) that precede slow
    GPU reads of host memory: huge-page splits, page migration, compaction."""
    out = {}
    try:
        for line in open("/proc/vmstat"):
            k, v = line.split()
            if k in VM_EVENTS:
                out[k] = int(v)
    except OSError:
        pass
    return out


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        v = float(json.load(open(p))["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------- CPU baseline

def oracle_layer_rate(w, host, seconds: float, max_layers: int | None = None):
    """Time the fp64 oracle (all steps) on whole layers of slot 0, using every
    host core, for about `seconds` (or max_layers layers).  Returns
    (layer-steps/s, cores, layers timed)."""
    import oracle
    cores = os.cpu_count() or 1
    os_ = oracle.Shape(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ctx_len, w.top_k,
                       w.window, w.dtype)
    orc = oracle.get()
    t0 = time.perf_counter()
    layers = 0
    while True:
        orc.layer(os_, host["q_spec"], host["q"], host["K"], host["V"], nthreads=cores)
        layers += 1
        el = time.perf_counter() - t0
        if (max_layers and layers >= max_layers) or (not max_layers and el >= seconds):
            break
    return layers / el, cores, layers


def host_slot(w, slot=0):
    """One layer slot on the host (plain memory) for the oracle."""
    dt = np.uint16 if w.dtype == synth.BF16 else np.float32
    q_spec = np.empty((w.batch, w.n_q_heads, w.head_dim), dt)
    q = np.empty_like(q_spec)
    K = np.empty((w.batch, w.n_kv_heads, w.ctx_len, w.head_dim), dt)
    V = np.empty_like(K)
    synth.fill_slot(w, slot, q_spec, q, K, V)
    return {"q_spec": q_spec, "q": q, "K": K, "V": V}


def config_of(w, args):
    return {"workload": w.name, "layers": w.n_layers, "distinct_layer_slots": w.n_slots,
            "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "ctx_len": w.ctx_len, "top_k": w.top_k, "window": w.window,
            "l2": "inputs larger than L2 (K of one layer is %.0f MiB; 129 MB L2)"
                  % (w.k_bytes() / 2**20),
            "parallelism": f"replicas x{args.gpus} (independent requests per GPU)",
            "gather_mode": ["bulk_copy", "load_store"][args.gather_mode],
            "gather_variant": getattr(args, "gather_chosen", None),
            "host_store": getattr(args, "store_used", args.host_alloc),
            "host_store_fill": getattr(args, "fill_used", args.fill),
            "schedule": getattr(args, "schedule_chosen", args.schedule),
            "copy_stream_priority": args.copy_priority,
            "correct_misses": bool(args.correct_misses),
            "landmark_chunk": args.landmarks or None,
            "topk": "fused into scoring" if args.fused_topk else "separate kernel"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one whole layer of slot 0."""
    if rank != 0:
        return
    w = workload(args)
    host = host_slot(w)
    cores = os.cpu_count() or 1
    oracle_layer_rate(w, host, 0, max_layers=max(1, args.warmup))
    rate, cores, layers = oracle_layer_rate(w, host, 0, max_layers=max(1, args.steps))
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 / rate, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args),
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{layers} whole layers of layer slot 0 (all "
                                   f"{w.units} (request, KV head) units), fp64 C oracle"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm

class HostStore:
    """The layer slots' host KV store: separate K and V stores [D][B][H_kv][n][d]
    or one interleaved store [D][B][H_kv][n][2][d] (each position's K row then
    its V row), in driver-allocated page-locked memory, locked huge pages or
    torch pinned memory."""

    def __init__(self, dd, kind, layout, shape5, dt):
        self.dd, self.kind, self.inter = dd, kind, layout == "interleaved"
        D, B, Hkv, n, d = shape5

        def alloc(shp):
            if kind in ("huge", "pinned"):
                return dd.host_empty(shp, dt, kind=kind)
            return torch.empty(shp, dtype=dt, pin_memory=True)
        if self.inter:
            self.kv = alloc((D, B, Hkv, n, 2, d))
            self.K, self.V = self.kv[:, :, :, :, 0, :], self.kv[:, :, :, :, 1, :]
        else:
            self.kv = None
            self.K, self.V = alloc(shape5), alloc(shape5)
        self.bytes = 2 * self.K.numel() * self.K.element_size()

    def flat(self, s):
        """Slot s as one contiguous host tensor (the copy-engine probe's source)."""
        return (self.kv[s] if self.inter else self.K[s]).reshape(-1)

    def fill(self, w, qs_h, q_h, dev, device_fill):
        """Write every slot with the seeded generator.  Returns the device key
        cache and the device window V."""
        dd = self.dd
        D, B, Hkv, n, d = self.K.shape
        W = w.window
        dt = self.K.dtype
        K_d = torch.empty((D, B, Hkv, n, d), dtype=dt, device=dev)
        vwin_d = torch.empty((D, B, Hkv, W, d), dtype=dt, device=dev) if W > 0 else None
        if not device_fill and not self.inter:
            for s in range(D):
                synth.fill_slot(w, s, qs_h[s], q_h[s], self.K[s], self.V[s])
                K_d[s].copy_(self.K[s])
                if W > 0:
                    vwin_d[s].copy_(self.V[s, :, :, n - W:, :])
            return K_d, vwin_d
        # Through page-locked staging: the interleaved store is written by
        # strided copies, and a device fill (as a KV offload writes the store)
        # by device-to-host copies.
        K_st = torch.empty((B, Hkv, n, d), dtype=dt, pin_memory=True)
        V_st = torch.empty((B, Hkv, n, d), dtype=dt, pin_memory=True)
        v_tmp = torch.empty((B, Hkv, n, d), dtype=dt, device=dev) if device_fill else None
        for s in range(D):
            synth.fill_slot(w, s, qs_h[s], q_h[s], K_st, V_st)
            K_d[s].copy_(K_st)
            if device_fill:
                v_tmp.copy_(V_st)
                self.K[s].copy_(K_d[s])
                self.V[s].copy_(v_tmp)
            else:
                self.K[s].copy_(K_st)
                self.V[s].copy_(V_st)
            if W > 0:
                vwin_d[s].copy_(V_st[:, :, n - W:, :])
        torch.cuda.synchronize()
        del K_st, V_st, v_tmp
        if hasattr(torch._C, "_host_emptyCache"):
            torch._C._host_emptyCache()
        return K_d, vwin_d

    def slot_host(self, s):
        """Slot s's K and V as contiguous host tensors (the oracle's inputs)."""
        return self.K[s].contiguous(), self.V[s].contiguous()

    def gather(self, shape, s, idx, kb, vb, mode=0, stream=None):
        if self.inter:
            self.dd.gather_h2d_kv(shape, self.kv[s], idx, kb, vb, mode=mode, stream=stream)
        else:
            self.dd.gather_h2d(shape, self.K[s], self.V[s], idx, kb, vb, mode=mode, stream=stream)

    def correct(self, shape, s, q, k_dev, idx_spec, kb_spec, vb_spec, idx_true, kb, vb, miss,
                mass, ws, stream=None):
        if self.inter:
            self.dd.correct_misses_kv(shape, q, k_dev, idx_spec, kb_spec, vb_spec, self.kv[s],
                                      idx_true, kb, vb, miss, mass, ws, stream=stream)
        else:
            self.dd.correct_misses(shape, q, k_dev, idx_spec, kb_spec, vb_spec, self.K[s],
                                   self.V[s], idx_true, kb, vb, miss, mass, ws, stream=stream)

    def io(self, s):
        """The host-store fields of a layer's LayerIO."""
        if self.inter:
            return dict(k_host=None, v_host=None, kv_host=self.kv[s])
        return dict(k_host=self.K[s], v_host=self.V[s], kv_host=None)

    def locked(self):
        return self.dd.host_store_locked(self.kv if self.inter else self.K) \
            if self.kind == "huge" else None


def run_ours(args, rank, world):
    import sparse_kv_prefetch_gb300 as dd

    w = workload(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    dt = torch.bfloat16 if w.dtype == synth.BF16 else torch.float32
    B, Hq, Hkv, d, n, k, W = (w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ctx_len,
                              w.top_k, w.window)
    D, L = w.n_slots, w.n_layers

    # Host store and the device-resident key cache, per layer slot.  The
    # store defaults to driver-allocated page-locked memory, which the host
    # never moved in any run; huge pages gather faster while the host leaves
    # them alone, but on many hosts it split and moved them, even minutes
    # into a run (see dd.h).
    huge0 = anon_huge_bytes()
    store_kind = "huge" if args.host_alloc == "auto" else args.host_alloc
    store = HostStore(dd, store_kind, args.host_layout, (D, B, Hkv, n, d), dt)
    store_bytes = store.bytes
    huge_frac = (anon_huge_bytes() - huge0) / store_bytes if huge0 is not None else None
    qs_h = torch.empty((D, B, Hq, d), dtype=dt, pin_memory=True)
    q_h = torch.empty((D, B, Hq, d), dtype=dt, pin_memory=True)
    t_gen = time.perf_counter()
    fill = args.fill if args.fill != "auto" else "cpu"
    args.fill_used = fill
    K_d, vwin_d = store.fill(w, qs_h, q_h, dev, fill == "device")
    t_gen = time.perf_counter() - t_gen
    qs_d, q_d = qs_h.to(dev), q_h.to(dev)
    outs = torch.empty((L, B, Hq, d), dtype=torch.float32, device=dev)

    shape = dd.Shape(B, Hq, Hkv, d, n, k, W, w.dtype)
    args.score_tc = dd.score_tensor_cores(shape) and not args.landmarks
    ctx = dd.Ctx(shape)
    late = bool(args.late_gather) or args.schedule == "late"
    pipe = args.schedule == "pipeline"
    guard = args.schedule == "guarded"
    if args.copy_priority == "high":
        compute, copy = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    else:
        compute, copy = torch.cuda.Stream(priority=-1), torch.cuda.Stream()
    sched_copy = None if args.schedule == "serial" else copy  # None: one stream
    C = args.landmarks
    lm_d = None
    if C:  # chunk landmarks of every layer slot, built once (prefill-time work)
        M = (n - W) // C
        lm_d = torch.empty((D, B, Hkv, M, d), dtype=torch.float32, device=dev)
        for s_ in range(D):
            dd.build_landmarks(shape, C, K_d[s_], lm_d[s_])
        ctx.set_landmark_chunk(C)
    torch.cuda.synchronize()

    # Host-link probe: one large contiguous pinned H2D copy, median of 10.
    flat0 = store.flat(0)
    probe_bytes = min(1 << 30, flat0.numel() * flat0.element_size())
    src = flat0.view(torch.uint8)[:probe_bytes]
    del flat0
    dst = torch.empty(probe_bytes, dtype=torch.uint8, device=dev)
    probe = []
    for i in range(13):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        e1.synchronize()
        if i >= 3:
            probe.append(probe_bytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    probe_gbs = statistics.median(probe)
    del dst, src

    # The gather alone (no other kernel running), cycling over every layer
    # slot so that each call meets cold host pages, as inside a decode step.
    U = B * Hkv
    g_idx = torch.empty((D, U, k), dtype=torch.int32, device=dev)
    g_sel = torch.empty((U, k), dtype=torch.float32, device=dev)
    g_lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    g_ws = torch.empty(dd.workspace_size(shape), dtype=torch.uint8, device=dev)
    g_kb = torch.empty((U, k, d), dtype=dt, device=dev)
    g_vb = torch.empty_like(g_kb)
    if C:
        lm_ws = torch.empty(dd.landmarks_workspace_size(shape, C), dtype=torch.uint8, device=dev)
        g_csel = torch.empty((U, k // C), dtype=torch.float32, device=dev)
    for s_ in range(D):
        if C:
            dd.score_topk_landmarks(shape, C, qs_d[s_], lm_d[s_], g_idx[s_], g_csel,
                                    g_lse, lm_ws, stream=compute)
        else:
            dd.score_topk(shape, qs_d[s_], K_d[s_], g_idx[s_], g_sel, g_lse, g_ws,
                          stream=compute)
    # Host-link steady state.  On this kind of host, periods of host-side
    # memory management (huge pages split, pages migrated) slow every GPU read
    # of a huge-page store ten-fold or more, for seconds to minutes.  Before
    # measuring, rounds of single-layer gathers (one per layer slot) run back
    # to back until two rounds in a row agree within 10 % and reach a floor:
    # 45 % of the copy probe for a huge-page store (a healthy one gathers at
    # 0.5-0.9 of it, a collapsed one at 0.005-0.05), 25 % otherwise (stores of
    # small pages are translation-bound well below the probe).  No pauses between rounds: after an idle spell the
    # first gathers over small pages run with cold translations.
    def settle(floor, max_s):
        t0 = time.perf_counter()
        rounds, rates, good = 0, [], 0
        # (A round of a small workload is launch-bound: its rate says nothing.)
        while w.gather_bytes() * D >= (64 << 20):
            evs = []
            for i in range(D):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(compute)
                store.gather(shape, i % D, g_idx[i % D], g_kb, g_vb, stream=compute)
                e1.record(compute)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            gbs = w.gather_bytes() / (statistics.median(a_.elapsed_time(b_) for a_, b_ in evs)
                                      * 1e-3) / 1e9
            rounds += 1
            ok = gbs >= floor * probe_gbs and bool(rates) and abs(gbs - rates[-1]) <= 0.1 * gbs
            rates.append(round(gbs, 1))
            good = good + 1 if ok else 0
            if good >= 1 or time.perf_counter() - t0 > max_s:
                break
        return {"settle_s": time.perf_counter() - t0, "settle_rounds": rounds,
                "settled": good >= 1 if rounds else None, "last_round_median_gbs": rates[-4:]}

    host_link = settle(0.45 if store_kind == "huge" else 0.25, args.settle_seconds)
    store_note = store_kind
    if args.host_alloc == "auto" and host_link["settled"] is False:
        # The huge-page store did not reach steady state: free it and write
        # the same (seeded) data into driver-allocated page-locked memory.
        import gc
        del store
        gc.collect()
        store = HostStore(dd, "pinned", args.host_layout, (D, B, Hkv, n, d), dt)
        t_refill = time.perf_counter()
        store.fill(w, qs_h, q_h, dev, fill == "device")
        t_gen += time.perf_counter() - t_refill
        store_kind = "pinned"
        store_note = ("pinned (the huge-page store did not settle within %.0f s; last rounds %s "
                      "GB/s)" % (host_link["settle_s"], host_link["last_round_median_gbs"]))
        host_link = settle(0.25, args.settle_seconds)
    args.store_used = store_note

    gather_alone = {}
    for mode in (0, 1):
        for i in range(2 * D):
            store.gather(shape, i % D, g_idx[i % D], g_kb, g_vb, mode=mode, stream=compute)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(compute)
        for i in range(4 * D):
            store.gather(shape, i % D, g_idx[i % D], g_kb, g_vb, mode=mode, stream=compute)
        e1.record(compute)
        e1.synchronize()
        gather_alone[mode] = w.gather_bytes() * 4 * D / (e0.elapsed_time(e1) * 1e-3) / 1e9

    # Predictability: for every layer slot, the rows prefetched with q_spec
    # against the real query's own top-k (dd_correct_misses).
    pred_miss, pred_mass = [], []
    if k <= 4096:
        c_idx = torch.empty((U, k), dtype=torch.int32, device=dev)
        c_kb, c_vb = torch.empty_like(g_kb), torch.empty_like(g_vb)
        c_miss = torch.empty(U, dtype=torch.int32, device=dev)
        c_mass = torch.empty((U, 2), dtype=torch.float32, device=dev)
        for s_ in range(D):
            store.gather(shape, s_, g_idx[s_], g_kb, g_vb, stream=compute)
            store.correct(shape, s_, q_d[s_], K_d[s_], g_idx[s_], g_kb, g_vb, c_idx, c_kb, c_vb,
                          c_miss, c_mass, g_ws, stream=compute)
            compute.synchronize()
            pred_miss.append(c_miss.cpu().numpy().copy())
            pred_mass.append(c_mass.cpu().numpy().copy())
        # Recall as a function of the speculation noise: q = q_spec + sigma N(0, 1)
        # (seeded, rounded to the stored dtype), on the first two layer slots.
        pred_sigma = {}
        gen = torch.Generator(device=dev)
        for sigma in (0.0, 0.05, 0.1, 0.2, 0.4, 0.8):
            gen.manual_seed(4321)
            miss = []
            for s_ in range(min(D, 2)):
                q_sig = (qs_d[s_].float() + sigma * torch.randn(
                    qs_d[s_].shape, generator=gen, device=dev)).to(dt)
                store.gather(shape, s_, g_idx[s_], g_kb, g_vb, stream=compute)
                store.correct(shape, s_, q_sig, K_d[s_], g_idx[s_], g_kb, g_vb, c_idx, c_kb,
                              c_vb, c_miss, c_mass, g_ws, stream=compute)
                compute.synchronize()
                miss.append(c_miss.cpu().numpy().copy())
            pred_sigma[str(sigma)] = float(1.0 - np.mean(miss) / k)
        del c_kb, c_vb
    predictability = None
    if pred_miss:
        pm, ms = np.stack(pred_miss), np.stack(pred_mass)
        predictability = {
            "recall": float(1.0 - pm.mean() / k),
            "recall_min_unit": float(1.0 - pm.max() / k),
            "mass_recall": float(ms[..., 0].sum() / ms[..., 1].sum()),
            "what": ("|TopK(q_spec) & TopK(q)| / k" if not C else
                     "|chunk rows selected with q_spec & TopK(q)| / k")
                    + " and the real query's selection score captured by the prefetched rows,"
                      " over all layer slots and units",
            "recall_vs_sigma": pred_sigma,
            "recall_vs_sigma_what": "q = q_spec + sigma N(0,1) drawn on the device, layer "
                                    "slots 0-1, all units",
        }
    del g_ws, g_kb, g_vb

    # Device residency of the step.  With landmarks the key cache itself is
    # not needed: the selection reads the landmarks and the attention reads
    # the window's keys from their own buffer.
    kwin_d = None
    if C:
        kwin_d = K_d[:, :, :, n - W:, :].contiguous() if W > 0 else None
        K_d = None  # frees the key cache
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        resident = lm_d.numel() * 4 + (2 * kwin_d.numel() * kwin_d.element_size() if W else 0)
    else:
        resident = K_d.numel() * K_d.element_size() + (
            vwin_d.numel() * vwin_d.element_size() if W else 0)

    def layer_io(l, qs, q):
        h = store.io(l % D)
        if C:
            return dd.LayerIO(qs, q, None, h["k_host"], h["v_host"],
                              vwin_d[l % D] if W > 0 else None, outs[l], lm_d[l % D],
                              kwin_d[l % D] if W > 0 else None, h["kv_host"])
        return dd.LayerIO(qs, q, K_d[l % D], h["k_host"], h["v_host"],
                          vwin_d[l % D] if W > 0 else None, outs[l], kv_host=h["kv_host"])

    layers = dd.Ctx.pack([layer_io(l, qs_d[l % D], q_d[l % D]) for l in range(L)])

    def step(copy_stream, timing=True):
        ctx.decode_step(layers, compute=compute, copy=copy_stream, timing=timing,
                        late_gather=late, pipeline=pipe, gather_mode=args.gather_mode,
                        correct_misses=args.correct_misses, landmarks=bool(C),
                        fused_topk=args.fused_topk, guarded=guard)

    def recorded(n_steps):
        """Phase times and per-layer scoring times of the last n timed steps,
        read after they ran (the events of every step stay in the context's
        ring, so the timed steps are enqueued back to back)."""
        ts = [ctx.timings(back=i) for i in reversed(range(n_steps))]
        sc = [x for i in reversed(range(n_steps)) for x in ctx.score_times(L, back=i)]
        return ts, sc

    compute.wait_stream(torch.cuda.current_stream())
    for _ in range(max(3, args.warmup)):
        step(sched_copy)
    torch.cuda.synchronize()
    if args.schedule == "auto":
        # Calibration: each two-stream schedule and the serial one in turn,
        # 3 steps each, twice.
        base = (("overlap", copy, False, False), ("serial", None, False, False),
                ("pipeline", copy, True, False), ("guarded", copy, False, True))
        if args.correct_misses:  # the pipeline schedule does not take miss correction
            base = tuple(b_ for b_ in base if b_[0] != "pipeline")
        variants = GATHER_VARIANTS if args.gather_auto else \
            tuple(v for v in GATHER_VARIANTS if v[1] == args.gather_mode)[:1]
        cands = tuple((name + "+" + vt, cs, pp, gg, vm, vg) for vt, vm, vg in variants
                      for name, cs, pp, gg in base)
        cal = {c[0]: 0.0 for c in cands}
        for _ in range(2):
            for name, cs, pp, gg, gm, geom in cands:
                pipe, guard = pp, gg  # read by step()
                args.gather_mode = gm
                set_gather_variant(dd, gm, geom)
                c0 = torch.cuda.Event(enable_timing=True)
                c1 = torch.cuda.Event(enable_timing=True)
                c0.record(compute)
                for _ in range(3):
                    step(cs, timing=False)
                c1.record(compute)
                torch.cuda.synchronize()
                cal[name] += c0.elapsed_time(c1) / 6
        names = [c[0] for c in cands]
        pick = min(cal, key=cal.get)
        if world > 1:  # every rank runs the same schedule: rank 0's choice
            import torch.distributed as dist
            t = torch.tensor([names.index(pick)], device=dev)
            dist.broadcast(t, 0)
            pick = names[int(t)]
        _, sched_copy, pipe, guard, args.gather_mode, geom = cands[names.index(pick)]
        set_gather_variant(dd, args.gather_mode, geom)
        args.gather_chosen = pick.split("+", 1)[1]
        args.schedule_chosen = (f"{pick} (auto; calibration ms per step: "
                                + ", ".join(f"{k} {v:.2f}" for k, v in cal.items()) + ")")
    n_phase = max(3, args.steps // 2)
    ctx.set_timing_depth(max(args.steps, n_phase))

    def region(copy_stream, n_steps, timing):
        """n_steps steps enqueued back to back; device ms on the compute stream."""
        torch.cuda.synchronize()
        r0 = torch.cuda.Event(enable_timing=True)
        r1 = torch.cuda.Event(enable_timing=True)
        r0.record(compute)
        for _ in range(n_steps):
            step(copy_stream, timing=timing)
        r1.record(compute)
        torch.cuda.synchronize()
        return r0.elapsed_time(r1)

    # Timed region: R back-to-back repeats of K steps with events around the
    # scoring phase only (for the roofline); value is the median repeat.
    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    vm0 = vm_events()
    repeats = max(1, args.repeats)
    region_ms, score_ms, launches = [], [], 0
    # An NVTX range marks the timed steps, so that a launch list can be taken
    # of them alone (ncu --nvtx --nvtx-include timed_steps/).
    torch.cuda.nvtx.range_push("timed_steps")
    for _ in range(repeats):
        barrier(world)
        region_ms.append(region(sched_copy, args.steps, "light"))
        barrier(world)
        timed, sc = recorded(args.steps)
        score_ms += sc
        launches = sum(t["launches"] for t in timed)
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    vm1 = vm_events()
    host_link["vm_events_in_timed_region"] = {k: vm1[k] - vm0.get(k, 0) for k in vm1
                                              if vm1[k] != vm0.get(k, 0)}
    region_s = [max_over_ranks(x * 1e-3, world) for x in region_ms]
    total_s = statistics.median(region_s)
    value = job_throughput(L, args.steps, total_s, world)
    values = [job_throughput(L, args.steps, x, world) for x in region_s]

    # Hidden fraction: the same steps with no per-layer events, overlapped (the
    # schedule timed above) and serial (one stream), interleaved, 3 each.
    t_over_l, t_ser_l = [], []
    for _ in range(3):
        t_over_l.append(region(sched_copy, args.steps, False) / args.steps)
        t_ser_l.append(region(None, args.steps, False) / args.steps)
    t_over, t_ser = statistics.median(t_over_l), statistics.median(t_ser_l)
    value_bare = job_throughput(L, args.steps, max_over_ranks(t_over * args.steps * 1e-3, world),
                                world)

    # The same steps as one CUDA graph launch each (captured once).
    ctx.capture_step(layers, compute, copy=sched_copy, late_gather=late, pipeline=pipe,
                     gather_mode=args.gather_mode, correct_misses=args.correct_misses,
                     landmarks=bool(C), fused_topk=args.fused_topk, guarded=guard)
    ctx.replay_step(compute)
    torch.cuda.synchronize()
    ev4, ev5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev4.record(compute)
    for _ in range(args.steps):
        ctx.replay_step(compute)
    ev5.record(compute)
    torch.cuda.synchronize()
    value_graph = job_throughput(L, args.steps,
                                 max_over_ranks(ev4.elapsed_time(ev5) * 1e-3, world), world)

    # Phase breakdown: steps with events around every phase, in the timed
    # schedule and serially (the serial gather time is the hidden fraction's
    # denominator).
    for _ in range(n_phase):
        step(sched_copy)
    torch.cuda.synchronize()
    phases, _ = recorded(n_phase)
    for _ in range(n_phase):
        step(None)
    torch.cuda.synchronize()
    serial, _ = recorded(n_phase)

    # End to end through the public API: per step copy every layer's q_spec and q
    # from pinned host memory, run the step, read every layer's output back.
    out_h = torch.empty((L, B, Hq, d), dtype=torch.float32, pin_memory=True)
    qs_l = torch.empty((L, B, Hq, d), dtype=dt, device=dev)
    q_l = torch.empty((L, B, Hq, d), dtype=dt, device=dev)
    qs_src = torch.stack([qs_h[l % D] for l in range(L)]).pin_memory()
    q_src = torch.stack([q_h[l % D] for l in range(L)]).pin_memory()
    layers_e2e = dd.Ctx.pack([layer_io(l, qs_l[l], q_l[l]) for l in range(L)])
    e2e_steps = max(3, args.steps // 2)

    def e2e_step():
        with torch.cuda.stream(compute):
            qs_l.copy_(qs_src, non_blocking=True)
            q_l.copy_(q_src, non_blocking=True)
        ctx.decode_step(layers_e2e, compute=compute, copy=sched_copy, late_gather=late,
                        pipeline=pipe,
                        gather_mode=args.gather_mode, correct_misses=args.correct_misses,
                        landmarks=bool(C), fused_topk=args.fused_topk, guarded=guard)
        with torch.cuda.stream(compute):
            out_h.copy_(outs, non_blocking=True)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(compute)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world)
    e2e_value = job_throughput(L, e2e_steps, e2e_s, world)
    if not torch.equal(out_h.to(dev), outs):
        raise RuntimeError("e2e read-back differs from the device outputs")

    # Derived rates.
    k_bytes, g_bytes = w.k_bytes(), w.gather_bytes()
    if C:  # the scoring phase reads the fp32 landmarks instead of K
        k_bytes = U * ((n - W) // C) * d * 4
    score_mean_ms = statistics.mean(score_ms)
    score_gbs = k_bytes / (score_mean_ms * 1e-3) / 1e9
    gather_ms_layer = statistics.mean(p["gather_ms"] for p in phases) / L
    gather_gbs = g_bytes / (gather_ms_layer * 1e-3) / 1e9
    g_ser = statistics.median(p["gather_ms"] for p in serial)
    comp_ser = statistics.median(p["score_ms"] + p["topk_ms"] + p["attn_ms"] for p in serial)
    hidden = max(0.0, min(1.0, (t_ser - t_over) / g_ser)) if g_ser > 0 else None
    peak, peak_kind = measured_hbm_peak()

    cpu = None
    if rank == 0 and world == 1 and not args.profile_case:
        K0_h, V0_h = store.slot_host(0)
        host = {"q_spec": qs_h[0], "q": q_h[0], "K": K0_h, "V": V0_h}
        rate, cores, nl = oracle_layer_rate(w, host, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{nl} whole layers of layer slot 0 (all {w.units} (request, KV head) "
                         f"units: scoring, full-sort top-k, attention) in fp64, "
                         f"~{args.cpu_seconds:.0f} s"}

    if rank != 0:
        ctx.close()
        return
    elt = 2 if w.dtype == synth.BF16 else 4
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": total_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == synth.BF16 else "f32",
        "data": "synthetic: seeded SplitMix64/Box-Muller K, V, q_spec ~ N(0,1), planted keys, "
                "q = q_spec + N(0, 0.1^2)",
        "config": config_of(w, args),
        "scoring_hbm_gbs": score_gbs,
        "scoring_serial_hbm_gbs": (k_bytes / (statistics.median(p["score_ms"] for p in serial)
                                              / L * 1e-3) / 1e9),
        "scoring_serial_what": "the same kernel in the phase-timed serial steps (no gather "
                               "beside it); scoring_hbm_gbs and roofline are inside the timed "
                               "schedule",
        "gather_host_link_gbs": gather_alone[0],
        "gather_frac_of_probe": gather_alone[0] / probe_gbs,
        "host_link_probe_gbs": probe_gbs,
        "gather_alone_gbs": {"bulk_copy": gather_alone[0], "load_store": gather_alone[1]},
        "gather_in_step_gbs": gather_gbs,
        "value_repeats": values,
        "value_min": min(values), "value_max": max(values),
        "value_spread": (max(values) - min(values)) / value,
        "value_what": f"median of {repeats} back-to-back regions of {args.steps} steps "
                      "(events around each layer's scoring only)",
        "hidden_fraction": hidden,
        "hidden_fraction_raw": (t_ser - t_over) / g_ser if g_ser > 0 else None,
        "hidden_fraction_what": "(serial - overlapped step time) / serial gather time; step "
                                "times from event-free regions of K steps, 3 of each schedule "
                                "interleaved (medians); gather time from phase-timed serial steps",
        "hidden_bound": min(1.0, comp_ser / g_ser) if g_ser > 0 else None,
        "overlapped_step_ms": t_over, "serial_step_ms": t_ser,
        "serial_gather_ms_per_step": g_ser,
        "phase_ms_per_step": {kk: statistics.mean(p[kk] for p in phases)
                              for kk in ("step_ms", "score_ms", "topk_ms", "gather_ms", "attn_ms")},
        "value_without_layer_events": value_bare,
        "value_without_layer_events_what": "the overlapped event-free regions of the hidden "
                                           "fraction (median)",
        "value_graph": value_graph,
        "value_graph_what": "the same K steps, each one launch of the step captured as a "
                            "CUDA graph (dd_ctx_capture_step / dd_ctx_replay_step)",
        "serial_phase_ms_per_step": {kk: statistics.mean(p[kk] for p in serial)
                                     for kk in ("step_ms", "score_ms", "topk_ms", "gather_ms",
                                                "attn_ms")},
        "roofline": {"bound": "hbm",
                     "kernel": ("score_kernel (top-k fused)" if args.fused_topk and not C
                                else "score_kernel" if not C else
                                "landmark selection phase (widen q, score, top-k, expand)"),
                     "achieved": score_gbs,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": score_gbs / peak,
                     "traffic": (None if args.profile_case or C
                                 else SCORE_TRAFFIC_BYTES.get((w.name, args.fused_topk))),
                     "algorithmic_bytes_per_launch": k_bytes,
                     "form": ("tensor cores (warp-level mma, fp32 accumulation)"
                              if args.score_tc else "per-lane fp32 FMA")},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": 2 * L * B * Hq * d * elt,
                "d2h_bytes_per_step": L * B * Hq * d * 4,
                "gather_host_bytes_per_step": L * g_bytes},
        "gpu_launches": launches,
        "predictability": predictability,
        "clocks": clk,
        "setup_s": {"generate": t_gen},
        "host_store": {"bytes": store_bytes, "huge_page_bytes": dd.host_page_bytes(),
                       "huge_page_fraction": huge_frac,
                       "kind": store_kind,
                       "locked": store.locked(),
                       "layout": args.host_layout},
        "host_link": host_link,
        "ctx_device_bytes": ctx.device_bytes,
        "hbm_resident_kv_bytes": resident,
        "hbm_resident_kv_what": ("fp32 landmarks + window K and V of every layer slot" if C else
                                 "key cache + window V of every layer slot"),
    }
    ctx.close()
    print(json.dumps(line), flush=True)


def main():
    args = resolve_defaults(parse())
    rank, world = dist_init(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
