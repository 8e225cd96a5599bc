"""Benchmark of the IBP gather-decompression hot path on GB300.

Default workload (the headline): sparse GNN features, 2,000,000 rows x 128
fp32 (512 B rows, 1 GB) compressed in place into pinned host slots (chunk
1 KB, Mask/Bitval from a 1 % sample at T = 0.95).  One step = one
ibp_gather_decompress of 200,000 uniform-random row ids: every stored byte is
read zero-copy over the host link by the kernel and 102.4 MB of rows are
written to HBM.

Reported (one JSON line on rank 0): delivered decompressed GB/s (value), its
fraction of the roofline min(HBM peak, link GB/s / ratio) where the link
bandwidth is measured in the same run by the aligned zero-copy copy kernel,
the end-to-end number through the C ABI with host buffers, the raw-gather
baseline, clocks, and the CPU oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload sparse|tiny|kv|dlrm|dense|weights|sweep|transfers|large|project]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2
PEAKS_FALLBACK = {"hbm_gbs": 6800.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": PEAKS_FALLBACK["hbm_gbs"], "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) over the timed region, plus one sample
    taken just before it starts and one just after it ends, so that a region
    shorter than the sampling period still carries a clock record."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def _once(self):
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                "--format=csv,noheader,nounits"], capture_output=True, text=True,
                               timeout=10)
            return [ln.strip() for ln in r.stdout.splitlines() if ln.strip()]
        except (OSError, subprocess.TimeoutExpired):
            return []

    def __enter__(self):
        self.lines.extend(self._once())  # edge sample: just before the region
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)
        self.lines.extend(self._once())  # edge sample: just after the region

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload setup
class SparseStore:
    """Sparse-GNN feature store compressed into pinned host slots by the GPU."""

    def __init__(self, torch, ibp, wl, dev, n_rows=2_000_000, dim=128, chunk=1024,
                 per_mille=10, num=95, den=100, seed=0, keep_raw=True):
        self.n_rows, self.R, self.C = n_rows, dim * 4, chunk
        t0 = time.time()
        rows = np.empty((n_rows, dim), np.float32)
        wl.sparse_gnn_rows(n_rows, dim, seed=seed, out=rows)
        log("generated %d x %d rows in %.1fs" % (n_rows, dim, time.time() - t0))
        self.rows_np = rows
        self.st = ibp.ibp_store_create(self.R, chunk, n_rows, 0)
        self.slot = ibp.ibp_store_get_info(self.st).slot_bytes
        self.slots = torch.empty((n_rows, self.slot), dtype=torch.uint8, pin_memory=True)
        d_rows = torch.from_numpy(rows.view(np.uint8)).to(dev)
        sample = wl.sample_ids(n_rows, per_mille, seed=seed)
        self.sample = sample
        d_sample = torch.from_numpy(sample).to(dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ibp.ibp_build_meta(self.st, d_rows, self.R, d_sample, len(sample), num, den)  # warm
        ev[0].record()
        ibp.ibp_build_meta(self.st, d_rows, self.R, d_sample, len(sample), num, den)
        ev[1].record()
        self.stored = torch.empty(n_rows, dtype=torch.int32, device=dev)
        ibp.ibp_compress(self.st, self.slots, d_rows, self.R, None, n_rows, self.stored)  # warm
        ev[2].record()
        ibp.ibp_compress(self.st, self.slots, d_rows, self.R, None, n_rows, self.stored)
        ev[3].record()
        torch.cuda.synchronize()
        t_meta = ev[0].elapsed_time(ev[1]) / 1e3
        t_comp = ev[2].elapsed_time(ev[3]) / 1e3
        # the companions on HBM-resident data: builder over all 2M rows (1 GB),
        # compressor into HBM slots (bound by HBM, not the host link)
        st2 = ibp.ibp_store_create(self.R, chunk, n_rows, 0)
        slots_dev = torch.empty((n_rows, self.slot), dtype=torch.uint8, device=dev)
        def med_time(fn, reps=5):  # median of `reps` timed calls after one warm-up
            fn()
            ts = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) / 1e3)
            return statistics.median(ts)

        t_meta_all = med_time(lambda: ibp.ibp_build_meta(st2, d_rows, self.R, None, n_rows, num,
                                                         den))
        torch.cuda.synchronize()  # the store's properties reach the host: specialised forms
        t_comp_hbm = med_time(lambda: ibp.ibp_compress(st2, slots_dev, d_rows, self.R, None,
                                                       n_rows, None))
        assert ibp.ibp_stream_status(st2, reset=True) == ibp.IBP_OK
        ibp.ibp_store_destroy(st2)
        del slots_dev
        self.companions = {
            "build_meta": {"rows": len(sample), "seconds": round(t_meta, 6),
                           "gbs": round(len(sample) * self.R / t_meta / 1e9, 2),
                           "note": "1% sample of rows in HBM, ones count + threshold + tables"},
            "compress": {"rows": n_rows, "seconds": round(t_comp, 6),
                         "gbs": round(n_rows * self.R / t_comp / 1e9, 2),
                         "note": "raw rows in HBM -> pinned host slots over the link"},
            "build_meta_all_rows_hbm": {"rows": n_rows, "seconds": round(t_meta_all, 6),
                                        "reps": "median of 5",
                                        "gbs": round(n_rows * self.R / t_meta_all / 1e9, 2),
                                        "note": "all 2M rows (1 GB) analysed, in HBM"},
            "compress_hbm": {"rows": n_rows, "seconds": round(t_comp_hbm, 6), "reps": "median of 5",
                             "gbs": round(n_rows * self.R / t_comp_hbm / 1e9, 2),
                             "note": "raw rows in HBM -> HBM slots (ratio 0.726: R read + "
                                     "stored written per row)"}}
        assert ibp.ibp_stream_status(self.st, reset=True) == ibp.IBP_OK
        self.raw_host = None
        if keep_raw:  # uncompressed host copy: the raw-gather baseline
            self.raw_host = torch.empty((n_rows, self.slot), dtype=torch.uint8, pin_memory=True)
            self.raw_host[:, :self.R].copy_(torch.from_numpy(rows.view(np.uint8)))
        del d_rows
        torch.cuda.empty_cache()
        self.stored_np = self.stored.cpu().numpy().astype(np.int64)
        log("store ready in %.1fs (ratio over all rows %.4f)" % (
            time.time() - t0, self.stored_np.sum() / (n_rows * self.R)))

    def close(self, ibp):
        ibp.ibp_store_destroy(self.st)


def cpu_oracle_decode(store, ids, mask, bitval, bitmap, threads):
    from oracle import ref_c
    slots = store.slots.numpy()
    out, bad = ref_c.decompress_batch(slots, bitmap, store.R, store.C, mask, bitval, ids=ids,
                                      slot_stride=store.slot, nthreads=threads)
    return out, bad


# ------------------------------------------------------------------ arms
def run_ours(args, rank, world, torch, dist):
    from lossless_invariant_bit_gb300 import dist as ibpdist
    from lossless_invariant_bit_gb300 import ibp
    from lossless_invariant_bit_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    store = SparseStore(torch, ibp, wl, dev, n_rows=args.rows, seed=args.seed)
    R, n = store.R, args.batch
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    # --- link probe: aligned zero-copy host -> HBM copy of 1 GB (best of 5)
    probe_bytes = (store.slots.numel() // 16) * 16
    probe_dst = torch.empty(probe_bytes, dtype=torch.uint8, device=dev)
    for _ in range(2):
        ibp.ibp_link_copy(probe_dst, store.slots, probe_bytes, sp)
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ibp.ibp_link_copy(probe_dst, store.slots, probe_bytes, sp)
        e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3
        best = t if best is None else min(best, t)
    link_gbs = probe_bytes / best / 1e9
    del probe_dst
    torch.cuda.empty_cache()
    log("link probe: %.1f GB/s host->HBM" % link_gbs)

    # --- a pool of distinct id batches, cycled (each rank its own: weak scaling)
    pool = min(args.pool, args.warmup + args.steps)
    ids_np = [wl.uniform_ids(n, store.n_rows, seed=args.seed, batch=ibpdist.batch_seed(rank, b))
              for b in range(pool)]
    ids_dev = [torch.from_numpy(x).to(dev) for x in ids_np]
    out = torch.empty((n, R), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ratios = [float(store.stored_np[x].sum()) / (n * R) for x in ids_np]

    def step_device(b):
        ibp.ibp_gather_decompress(store.st, out, store.slots, None, ids_dev[b % pool], n, sp)

    def timed(fn, steps_from, count, pre=None):
        evs = []
        for b in range(steps_from, steps_from + count):
            flush.zero_()  # L2 flush, outside the timed events
            if pre:
                pre(b)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(b)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(c) / 1e3 for a, c in evs]

    for b in range(args.warmup):
        step_device(b)
    torch.cuda.synchronize()
    assert ibp.ibp_stream_status(store.st, reset=True) == ibp.IBP_OK
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        times = timed(step_device, args.warmup, args.steps)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    assert ibp.ibp_stream_status(store.st, reset=True) == ibp.IBP_OK
    t_total = sum(times)
    t_total = ibpdist.max_over_ranks(t_total, dist, dev)
    rows_all = n * args.steps * world
    value = rows_all * R / t_total / 1e9
    t_launch = statistics.mean(times)
    ratio = statistics.mean(ratios[(args.warmup + b) % pool] for b in range(args.steps))

    # parity spot check of the last timed batch against the oracle (rows sampled)
    last = (args.warmup + args.steps - 1) % pool
    ibp.ibp_gather_decompress(store.st, out, store.slots, None, ids_dev[last], n, sp)
    torch.cuda.synchronize()
    pick = np.random.default_rng(1).choice(n, size=2000, replace=False)
    got = out[torch.from_numpy(pick).to(dev)].cpu().numpy()
    want = store.rows_np.view(np.uint8)[ids_np[last][pick]]
    parity_ok = bool(np.array_equal(got, want))

    # --- raw gather baseline (uncompressed rows over the same link)
    raw_times = timed(lambda b: ibp.ibp_gather_copy(out, store.raw_host, store.slot, R,
                                                    ids_dev[b % pool], n, store.n_rows, sp),
                      args.warmup, args.steps)
    raw_gbs = n * R * len(raw_times) / sum(raw_times) / 1e9

    # --- the same batches through the address-ordered gather (ids bucketed by
    # region first; identical output)
    ws = torch.empty(ibp.order_workspace_bytes(n), dtype=torch.uint8, device=dev)

    def step_ordered(b):
        ibp.ibp_gather_decompress_ordered(store.st, out, R, store.slots, None, ids_dev[b % pool],
                                          n, ws, ws.numel(), sp)

    osteps = min(args.steps, 200)
    for b in range(args.warmup):
        step_ordered(b)
    o_times = timed(step_ordered, args.warmup, osteps)
    assert ibp.ibp_stream_status(store.st, reset=True) == ibp.IBP_OK
    lasto = (args.warmup + osteps - 1) % pool
    o_ok = bool(np.array_equal(out[torch.from_numpy(pick).to(dev)].cpu().numpy(),
                               store.rows_np.view(np.uint8)[ids_np[lasto][pick]]))
    ordered_res = {"value": round(n * R / statistics.mean(o_times) / 1e9, 3), "unit": "GB/s",
                   "steps": osteps, "parity_sampled_rows_ok": o_ok,
                   "note": "ibp_gather_decompress_ordered on the same batches (four launches "
                           "per step)"}
    del ws

    # --- cache front: a quarter of the rows' stored slots also held in HBM; one
    # launch reads the hits from HBM and the misses over the link
    front = None
    if not args.no_cache_front:
        gf = np.random.default_rng(args.seed + 7)
        n_cache = store.n_rows // 4
        cached = np.sort(gf.choice(store.n_rows, size=n_cache, replace=False))
        cmap_np = np.full(store.n_rows, -1, np.int64)
        cmap_np[cached] = np.arange(n_cache)
        cache = store.slots[torch.from_numpy(cached)].to(dev)
        cmap_dev = torch.from_numpy(cmap_np).to(dev)

        def step_front(b):
            ibp.ibp_gather_decompress_cached(store.st, out, R, store.slots, cache, n_cache,
                                             cmap_dev, ids_dev[b % pool], n, sp)

        fsteps = min(args.steps, 200)
        for b in range(args.warmup):
            step_front(b)
        f_times = timed(step_front, args.warmup, fsteps)
        assert ibp.ibp_stream_status(store.st, reset=True) == ibp.IBP_OK
        f_launch = statistics.mean(f_times)
        f_val = n * R / f_launch / 1e9
        lastf = (args.warmup + fsteps - 1) % pool
        f_ok = bool(np.array_equal(out[torch.from_numpy(pick).to(dev)].cpu().numpy(),
                                   store.rows_np.view(np.uint8)[ids_np[lastf][pick]]))
        hits, link_ratio = [], []
        for b in range(fsteps):
            x = ids_np[(args.warmup + b) % pool]
            miss = cmap_np[x] < 0
            hits.append(1.0 - float(miss.mean()))
            link_ratio.append(float(store.stored_np[x[miss]].sum()) / (n * R))
        f_roof = min(peaks["hbm_gbs"], link_gbs / statistics.mean(link_ratio))
        front = {"value": round(f_val, 3), "unit": "GB/s", "steps": fsteps,
                 "cached_rows": n_cache, "hit_rate": round(statistics.mean(hits), 4),
                 "link_bytes_per_row_delivered": round(statistics.mean(link_ratio), 5),
                 "roofline_peak": round(f_roof, 2), "frac": round(f_val / f_roof, 4),
                 "speedup_vs_host_only": None, "parity_sampled_rows_ok": f_ok,
                 "note": "ibp_gather_decompress_cached: the stored slots of a seeded quarter "
                         "of the rows also in HBM (a cache map id -> cache slot); same id "
                         "batches; roofline = min(HBM, link / link bytes per delivered byte)"}
        del cache, cmap_dev
        torch.cuda.empty_cache()

    # --- end to end through the C ABI with host buffers: the ids, the compressed
    # store and the output all live in pinned host memory; the one call moves
    # ids + stored bytes host->GPU and the rows GPU->host inside its kernel
    ids_host = [torch.from_numpy(x).pin_memory() for x in ids_np]
    out_host = torch.empty((n, R), dtype=torch.uint8, pin_memory=True)

    def step_e2e(b):
        ibp.ibp_gather_decompress(store.st, out_host, store.slots, None, ids_host[b % pool], n, sp)

    for b in range(args.warmup):
        step_e2e(b)
    e2e_times = timed(step_e2e, args.warmup, args.steps)
    t_e2e = sum(e2e_times)
    t_e2e = ibpdist.max_over_ranks(t_e2e, dist, dev)
    e2e_gbs = n * R * args.steps * world / t_e2e / 1e9
    lastb = (args.warmup + args.steps - 1) % pool
    e2e_ok = bool(np.array_equal(out_host.numpy()[pick],
                                 store.rows_np.view(np.uint8)[ids_np[lastb][pick]]))
    e2e_h2d = int(statistics.mean(8 * n + float(store.stored_np[ids_np[(args.warmup + b) % pool]].sum())
                                  for b in range(args.steps)))

    # --- the dominant kernel's roofline
    hbm = peaks["hbm_gbs"]
    roof = min(hbm, link_gbs / ratio)
    delivered_per_launch = n * R / t_launch / 1e9
    algo_bytes = statistics.mean(float(store.stored_np[ids_np[(args.warmup + b) % pool]].sum())
                                 + n * R + 8 * n for b in range(args.steps))
    result = {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": round(value, 3),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_total / args.steps * 1e3, 4),
        "ms_per_step_median": round(statistics.median(times) * 1e3, 4),
        "ms_per_step_min": round(min(times) * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u32",
        "data": "synthetic (seeded numpy: sparse GNN features, 1.0 w.p. 0.01 else 0.0)",
        "config": {
            "workload": "sparse GNN gather-decompress: 2,000,000 x 128 fp32 rows in pinned "
                        "host slots, chunk 1 KB, 1% sample, T=0.95, batches of 200,000 "
                        "uniform ids",
            "rows": store.n_rows, "row_bytes": R, "chunk_bytes": store.C,
            "batch_ids": n, "distinct_batches": pool, "source": "pinned host (zero-copy)",
            "l2": "flushed between steps (256 MB write, outside the timed events)",
            "parallelism": "dp%d (id batches sharded, no collective)" % world,
        },
        "ratio": round(ratio, 5),
        "link_gbs": round(link_gbs, 2),
        "raw_gather_gbs": round(raw_gbs, 2),
        "speedup_vs_raw_gather": round(value / world / raw_gbs, 3),
        "parity_sampled_rows_ok": parity_ok,
        "roofline": {
            "bound": "link",
            "achieved": round(delivered_per_launch, 2),
            "peak": round(roof, 2),
            "unit": "GB/s",
            "frac": round(delivered_per_launch / roof, 4),
            # host-link read bytes of one 200,000-id launch: ncu capture of this kernel
            # (profiles/k_decode_gather_sparse_gnn.md), 18.93 MB per 50,000 ids x 4;
            # its DRAM bytes are ~0 there (the output is still in L2 at kernel end)
            "traffic": 75.7e6,
            "traffic_is": "host-link (sysmem) read bytes per launch from ncu, scaled "
                          "from a 50,000-id capture",
            "peak_is": "min(HBM %s %.0f GB/s, link %.1f GB/s measured in this run / ratio %.4f)"
                       % (peaks["source"], hbm, link_gbs, ratio),
            "kernel": "k_decode_fast<true, mode, small> (ibp_gather_decompress, host-memory source)",
            "algorithmic_bytes_per_launch": int(algo_bytes),
            "link_bytes_achieved_gbs": round(ratio * delivered_per_launch, 2),
        },
        "e2e": {"value": round(e2e_gbs, 3), "unit": "GB/s",
                "h2d_bytes_per_step": e2e_h2d, "d2h_bytes_per_step": n * R,
                "how": "ibp_gather_decompress with ids, compressed slots and output rows all "
                       "in pinned host memory: the kernel reads ids + stored bytes over the "
                       "link and writes the rows back over it (zero-copy both ways)",
                "parity_sampled_rows_ok": e2e_ok},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "companions": store.companions,
    }
    ordered_res["frac"] = round(ordered_res["value"] / roof, 4)
    result["ordered_gather"] = ordered_res
    if front is not None:
        front["speedup_vs_host_only"] = round(front["value"] / (value / world), 3)
        result["cache_front"] = front

    # --- CPU baseline: the oracle on the host cores, one batch (rank 0, N = 1)
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(store, ids_np, ibp)
        # the oracle's rows for 2000 ids of the last timed batch against the
        # GPU's, the generated rows and the oracle's compression of them
        leg = oracle_leg(ibp, store.st, store.slots, R, store.C, ids_np[last][pick], got, want)
        result["cpu_baseline"]["parity_oracle_ok"] = leg["parity_oracle_ok"]

    # --- the chunk-aware builder: the threshold chosen from the sample itself
    if not args.no_tuned:
        cands = [(3, 4), (85, 100), (9, 10), (95, 100), (97, 100), (99, 100), (999, 1000), (1, 1)]
        d_rows = torch.from_numpy(store.rows_np.view(np.uint8)).to(dev)
        d_sample = torch.from_numpy(store.sample).to(dev)
        chosen = torch.zeros(1, dtype=torch.int32, device=dev)
        ibp.ibp_build_meta_tuned(store.st, d_rows, R, d_sample, len(store.sample),
                                 [c[0] for c in cands], [c[1] for c in cands], chosen, None, sp)
        stored_t = torch.empty(store.n_rows, dtype=torch.int32, device=dev)
        ibp.ibp_compress(store.st, store.slots, d_rows, R, None, store.n_rows, stored_t, sp)
        torch.cuda.synchronize()
        assert ibp.ibp_stream_status(store.st, reset=True) == ibp.IBP_OK
        del d_rows
        st_np = stored_t.cpu().numpy().astype(np.int64)
        tsteps = min(args.steps, 200)
        for b in range(args.warmup):
            step_device(b)
        t_times = timed(step_device, args.warmup, tsteps)
        t_ratio = statistics.mean(float(st_np[ids_np[(args.warmup + b) % pool]].sum()) / (n * R)
                                  for b in range(tsteps))
        t_launch = statistics.mean(t_times)
        t_val = n * R / t_launch / 1e9
        t_roof = min(peaks["hbm_gbs"], link_gbs / t_ratio)
        got = out[torch.from_numpy(pick).to(dev)].cpu().numpy()
        lastt = (args.warmup + tsteps - 1) % pool
        want = store.rows_np.view(np.uint8)[ids_np[lastt][pick]]
        result["tuned_builder"] = {
            "candidates_T": ["%d/%d" % c for c in cands],
            "chosen_T": "%d/%d" % cands[int(chosen.item())],
            "ratio": round(t_ratio, 5), "value": round(t_val, 3), "unit": "GB/s",
            "steps": tsteps, "roofline_peak": round(t_roof, 2), "frac": round(t_val / t_roof, 4),
            "speedup_vs_raw_gather": round(t_val / raw_gbs, 3),
            "parity_sampled_rows_ok": bool(np.array_equal(got, want)),
            "note": "same rows and id batches; Mask/Bitval from ibp_build_meta_tuned on the "
                    "same 1% sample"}
    store.close(ibp)
    return result

def run_tiny(args, rank, world, torch, dist):
    """Cache path: full decompression of a packed HBM cache.  128 distinct
    replicas of the tiny workload (4096 x 256 fp32 each, 524,288 rows, 512 MB
    raw) so that one launch moves far more than the 129 MB L2; Mask/Bitval from
    replica 0 at T = 0.95, chunk 256 B."""
    from lossless_invariant_bit_gb300 import dist as ibpdist
    from lossless_invariant_bit_gb300 import ibp
    from lossless_invariant_bit_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    reps, per, R, C = args.replicas, 4096, 1024, 256
    n = reps * per
    rows = np.empty((n, 256), np.float32)
    for r in range(reps):
        rows[r * per:(r + 1) * per] = wl.tiny_rows(seed=args.seed + r)[0]
    rb = rows.view(np.uint8)
    st = ibp.ibp_store_create(R, C, n, R)
    d_rows = torch.from_numpy(rb).to(dev)
    ibp.ibp_build_meta(st, d_rows, R, None, per, 95, 100)
    slots = torch.empty((n, R), dtype=torch.uint8, device=dev)
    stored = torch.empty(n, dtype=torch.int32, device=dev)
    ibp.ibp_compress(st, slots, d_rows, R, None, n, stored)
    offs = torch.empty(n + 1, dtype=torch.int64, device=dev)
    ibp.ibp_pack(st, None, offs, slots, stored, n)
    total = int(offs[-1].item())
    cache = torch.empty(total, dtype=torch.uint8, device=dev)
    ibp.ibp_pack(st, cache, offs, slots, stored, n)
    torch.cuda.synchronize()
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    del slots
    stored_sum = int(stored.sum().item())
    ratio = stored_sum / (n * R)
    out = torch.empty((n, R), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def step(_):
        ibp.ibp_decompress(st, out, cache, offs, n, sp)

    def timed(fn, count):
        # no L2 flush: each step reads the whole packed cache and writes all
        # rows (>= 173 MB + 537 MB at 128 replicas, far above the 129 MB L2),
        # and a flush's dirty lines would be written back inside the next step
        evs = []
        for b in range(count):
            if args.replicas < 64:
                flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(b)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(c) / 1e3 for a, c in evs]

    for b in range(args.warmup):
        step(b)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    with ClockSampler(dev.index) as clk:
        times = timed(step, args.steps)
    if dist:
        dist.barrier()
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    parity_ok = bool(torch.equal(out, d_rows))
    # cpu_baseline leg: the oracle decodes the first 8192 rows (two replicas)
    # from a host copy of the packed cache; its rows against the GPU's
    from oracle import ref_c
    k_or = 2 * per
    mask = np.zeros(R // 4, np.uint32)
    bitval = np.zeros(R // 4, np.uint32)
    ibp.ibp_meta_get(st, mask, bitval)
    bitmap = np.zeros((n + 31) // 32, np.uint32)
    ibp.ibp_bitmap_get(st, bitmap)
    offs_np = offs[:k_or + 1].cpu().numpy().view(np.uint64)
    cache_np = cache[:int(offs_np[-1]) + R].cpu().numpy()
    threads = len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    orows, obad = ref_c.decompress_batch(cache_np, bitmap, R, C, mask, bitval, n=k_or,
                                         offsets=offs_np[:k_or], nthreads=threads)
    t_or = time.perf_counter() - t0
    leg = {"value": round(k_or * R / t_or / 1e9, 4), "unit": "GB/s", "cores": threads,
           "kind": "oracle",
           "sample": "the first %d rows of the packed cache decoded by the oracle C decoder "
                     "(OpenMP over rows, %.2f s)" % (k_or, t_or),
           "parity_oracle_ok": bool(obad == 0 and np.array_equal(orows, out[:k_or].cpu().numpy())
                                    and np.array_equal(orows, rb[:k_or]))}
    t_total = sum(times)
    t_total = ibpdist.max_over_ranks(t_total, dist, dev)
    value = n * R * args.steps * world / t_total / 1e9
    t_launch = statistics.mean(times)
    hbm = peaks["hbm_gbs"]
    moved = (stored_sum + n * R) / t_launch / 1e9  # read stored + write rows

    # single-batch latency: one replica (4096 rows, 4 MB: L2-resident, launch-bound)
    lat = []
    for b in range(23):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ibp.ibp_decompress(st, out, cache, offs, per, sp)
        e1.record(stream)
        e1.synchronize()
        if b >= 3:
            lat.append(e0.elapsed_time(e1) * 1e3)

    # e2e: packed cache in HBM, output read back to pinned host each step
    out_host = torch.empty((n, R), dtype=torch.uint8, pin_memory=True)

    def step_e2e(b):  # the call with a host output buffer: rows written over the link
        ibp.ibp_decompress(st, out_host, cache, offs, n, sp)

    step_e2e(0)
    e2e_t = sum(timed(step_e2e, max(3, min(args.steps, 50))))
    e2e_steps = max(3, min(args.steps, 50))
    res = {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_total / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded numpy: tiny workload, 1 + k/1024 fp32, 1% N(0,1) rows)",
        "config": {"workload": "tiny cache path: %d distinct replicas of 4096 x 256 fp32 rows "
                               "(%d rows), packed HBM cache, chunk 256 B, T=0.95, full "
                               "decompress" % (reps, n),
                   "rows": n, "row_bytes": R, "chunk_bytes": C, "source": "HBM packed cache",
                   "l2": ("inputs larger than L2: every step reads the %.0f MB packed cache and "
                          "writes %.0f MB of rows; no flush" % (total / 1e6, n * R / 1e6))
                         if reps >= 64 else "flushed between steps (256 MB write, outside the "
                                            "timed events)",
                   "parallelism": "dp%d (replicas, no collective)" % world},
        "ratio": round(ratio, 5),
        "parity_all_rows_ok": parity_ok,
        "single_batch_us": {"median": round(statistics.median(lat), 2), "min": round(min(lat), 2),
                            "rows": per},
        "roofline": {"bound": "hbm", "achieved": round(moved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(moved / hbm, 4),
                     # dram read + write of a 48-replica launch (profiles/
                     # k_decode_tiles_tiny_cache.md) scaled to this launch's rows
                     "traffic": round(210.11e6 * n / (48 * 4096)),
                     "traffic_is": "dram__bytes_read.sum + dram__bytes_write.sum from ncu, "
                                   "scaled from a 196,608-row capture (part of the output is "
                                   "still in L2 when the kernel ends)",
                     "peak_is": "HBM copy bandwidth, %s" % peaks["source"],
                     "kernel": "k_decode_tiles<uniform1> (ibp_decompress, packed offsets: "
                               "bulk copies of 32-row tiles)",
                     "algorithmic_bytes_per_launch": int(stored_sum + n * R + 8 * n)},
        "e2e": {"value": round(n * R * e2e_steps / e2e_t / 1e9, 3), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": n * R},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": leg,
    }
    ibp.ibp_store_destroy(st)
    return res


def run_kv(args, rank, world, torch, dist):
    """LLM KV-cache fetch, OPT-6.7B shape: 32 layers x {K, V}, batch 20, 2048
    token slots, 32 heads x 128 fp16 = 8 KB rows (21.5 GB of pinned host
    slots).  K/V ~ N(0,1) x per-channel log-normal scale, 2 % outlier channels
    x20, generated on the GPU (seeded torch generator per layer and K|V).
    Mask/Bitval per (layer, K|V) from its 20 x 1920 prompt rows, chunk 256 B
    (one head).  A step is one decode step's re-fetch: for each of the 64
    (layer, K|V) stores, gather the 20 x (1920 + s) rows of the history into
    HBM (s = 0)."""
    from lossless_invariant_bit_gb300 import dist as ibpdist
    from lossless_invariant_bit_gb300 import ibp

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    # one step moves ~20 GB over the host link (~0.1 s): at most 20 timed steps
    args = argparse.Namespace(**vars(args))
    args.steps, args.warmup = min(args.steps, 20), min(args.warmup, 3)
    L, B, T, P, CH = args.kv_layers, 20, 2048, 1920, 4096
    R, C = CH * 2, 256
    rows_per = B * T
    t0 = time.time()
    stores, slots = [], []
    g = torch.Generator(device=dev)
    ratio_num = 0
    prompt_ids = torch.from_numpy(
        (np.arange(B)[:, None] * T + np.arange(P)[None, :]).reshape(-1).astype(np.int64)).to(dev)
    check = None
    kv_lengths = []  # each store's stored sizes, attached to it
    newrows = []  # rows of the decode tokens 1920..2047, kept on the GPU for the decode steps
    for layer in range(L):
        for kv in range(2):
            g.manual_seed(args.seed * 1000003 + layer * 2 + kv)
            z = torch.randn(CH, generator=g, device=dev)
            scale = torch.exp(0.5 * z)
            out_ch = torch.randperm(CH, generator=g, device=dev)[:int(round(0.02 * CH))]
            scale[out_ch] *= 20.0
            x = (torch.randn((rows_per, CH), generator=g, device=dev) * scale).to(torch.float16)
            xb = x.view(torch.uint8)
            st = ibp.ibp_store_create(R, C, rows_per, R)
            ibp.ibp_build_meta(st, xb, R, prompt_ids, len(prompt_ids), 95, 100)
            sl = torch.empty((rows_per, R), dtype=torch.uint8, pin_memory=True)
            stored = torch.empty(rows_per, dtype=torch.int32, device=dev)
            ibp.ibp_compress(st, sl, xb, R, None, rows_per, stored)
            ratio_num += int(stored[:].view(B, T)[:, :P].sum().item())
            ibp.ibp_store_set_lengths(st, stored)  # kept current by the decode-step compress
            kv_lengths.append(stored)
            if layer == 0 and kv == 0:
                check = xb.view(B, T, R)[:, :P].clone()
            newrows.append(xb.view(B, T, R)[:, P:].clone())
            stores.append(st)
            slots.append(sl)
            del x, xb
    torch.cuda.synchronize()
    log("KV store ready in %.1fs" % (time.time() - t0))
    ratio = ratio_num / (2 * L * B * P * R)
    ids = prompt_ids  # history at decode step 0: the 1920 prompt tokens
    n = len(ids)
    out = torch.empty((B, P, R), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def step(_):
        for st, sl in zip(stores, slots):
            ibp.ibp_gather_decompress(st, out, sl, None, ids, n, sp)

    for b in range(args.warmup):
        step(b)
    torch.cuda.synchronize()
    ibp.ibp_gather_decompress(stores[0], out, slots[0], None, ids, n, sp)
    torch.cuda.synchronize()
    parity_ok = bool(torch.equal(out, check))
    # cpu_baseline leg: the oracle decodes 2048 sampled rows of layer 0's K
    # store from the same host slots (its rows against the GPU's and the
    # generated ones; its compression against the stored bytes)
    pick = np.sort(np.random.default_rng(3).choice(n, 2048, replace=False))
    ids_np = prompt_ids.cpu().numpy()
    leg = oracle_leg(ibp, stores[0], slots[0], R, C, ids_np[pick],
                     out.view(-1, R)[torch.from_numpy(pick).to(dev)].cpu().numpy(),
                     check.reshape(-1, R)[torch.from_numpy(pick).to(dev)].cpu().numpy(),
                     note="; layer 0 K store, prompt rows")
    evs = []
    with ClockSampler(dev.index) as clk:
        for b in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step(b)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
    for st in stores:
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    times = [a.elapsed_time(c) / 1e3 for a, c in evs]
    t_total = ibpdist.max_over_ranks(sum(times), dist, dev)
    raw_bytes = 2 * L * n * R
    value = raw_bytes * args.steps * world / t_total / 1e9
    pbytes = (slots[0].numel() // 16) * 16  # one store's slots, 335 MB
    probe = torch.empty(pbytes, dtype=torch.uint8, device=dev)
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ibp.ibp_link_copy(probe, slots[0], pbytes, sp)
        e1.record(stream)
        e1.synchronize()
        tt = e0.elapsed_time(e1) / 1e3
        best = tt if best is None else min(best, tt)
    link = pbytes / best / 1e9
    del probe
    roof = min(measured_peaks()["hbm_gbs"], link / ratio)

    # the same fetch decompressed straight into the attention layout
    # [B, H, P, D] (ibp_gather_decompress_split: each 256-byte head to its own row)
    H, D = 32, 128
    att = torch.empty((B, H, P, D * 2), dtype=torch.uint8, device=dev)

    def step_att(_):
        for st, sl in zip(stores, slots):
            ibp.ibp_gather_decompress_split(st, att, P, H * P * D * 2, D * 2, P * D * 2, sl, None,
                                            ids, n, sp)

    step_att(0)
    ibp.ibp_gather_decompress_split(stores[0], att, P, H * P * D * 2, D * 2, P * D * 2, slots[0],
                                    None, ids, n, sp)
    torch.cuda.synchronize()
    att_ok = bool(torch.equal(att, check.view(B, P, H, D * 2).permute(0, 2, 1, 3)))
    asteps = min(args.steps, 10)
    aev = []
    for b in range(asteps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step_att(b)
        e1.record(stream)
        aev.append((e0, e1))
    torch.cuda.synchronize()
    for st in stores:
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    t_att = sum(a.elapsed_time(c) / 1e3 for a, c in aev)
    att_gbs = 2 * L * n * R * asteps / t_att / 1e9
    del att

    # decode steps: each compresses the 20 new rows of every (layer, K|V) into
    # their host slots (1280 rows), then re-fetches the whole history
    decode = []
    stored1 = torch.empty(B, dtype=torch.int32, device=dev)
    for s_ in (0, 63, 127):
        tok = P + s_
        sids = torch.from_numpy((np.arange(B) * T + tok).astype(np.int64)).to(dev)
        hist = torch.from_numpy((np.arange(B)[:, None] * T + np.arange(tok + 1)[None, :])
                                .reshape(-1).astype(np.int64)).to(dev)
        nh = len(hist)
        outh = torch.empty((nh, R), dtype=torch.uint8, device=dev)

        def comp(stream_handle=sp):
            for st, sl, nr in zip(stores, slots, newrows):
                ibp.ibp_compress(st, sl, nr[:, s_], (T - P) * R, sids, B, stored1, stream_handle)

        def fetch():
            for st, sl in zip(stores, slots):
                ibp.ibp_gather_decompress(st, outh, sl, None, hist, nh, sp)

        tc, tf = [], []
        for rep_ in range(4):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(stream)
            comp()
            e[1].record(stream)
            fetch()
            e[2].record(stream)
            torch.cuda.synchronize()
            if rep_:  # the first is a warm-up
                tc.append(e[0].elapsed_time(e[1]) / 1e3)
                tf.append(e[1].elapsed_time(e[2]) / 1e3)
        # the same 64 compress calls replayed from one CUDA graph
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph):
            comp(torch.cuda.current_stream().cuda_stream)
        tgr = []
        for rep_ in range(4):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record(stream)
            gph.replay()
            e[1].record(stream)
            torch.cuda.synchronize()
            if rep_:
                tgr.append(e[0].elapsed_time(e[1]) / 1e3)
        del gph
        for st in stores:
            assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
        ibp.ibp_gather_decompress(stores[0], outh, slots[0], None, hist, nh, sp)
        torch.cuda.synchronize()
        got = outh.view(B, tok + 1, R)
        ok = bool(torch.equal(got[:, :P], check) and torch.equal(got[:, P:], newrows[0][:, :s_ + 1]))
        decode.append({"step": s_, "history_rows_per_store": nh,
                       "compress_us": round(statistics.median(tc) * 1e6, 1),
                       "compress_us_cuda_graph": round(statistics.median(tgr) * 1e6, 1),
                       "compress_gbs": round(2 * L * B * R / statistics.median(tc) / 1e9, 2),
                       "fetch_gbs": round(2 * L * nh * R / statistics.median(tf) / 1e9, 2),
                       "parity_layer0_ok": ok})
        del outh
    del newrows
    proj = kv_decode_projection(torch, ibp, dev, stream, sp, seed=args.seed)
    res = {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_total / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded torch generator on the GPU: OPT-6.7B-shaped K/V)",
        "config": {"workload": "KV-cache fetch: %d layers x {K,V}, batch 20, 1920 prompt "
                               "tokens of 2048 slots, 8 KB fp16 rows in pinned host slots, "
                               "chunk 256 B, T=0.95; one step = 64 per-layer gathers" % L,
                   "rows_per_store": rows_per, "row_bytes": R, "chunk_bytes": C,
                   "l2": "flushed between steps (256 MB write, outside the timed events)"},
        "ratio": round(ratio, 5), "link_gbs": round(link, 2), "parity_layer0_ok": parity_ok,
        "roofline": {"bound": "link", "achieved": round(value / world, 2), "peak": round(roof, 2),
                     "unit": "GB/s", "frac": round(value / world / roof, 4),
                     # host-link read sectors of one (layer, K|V) fetch of 38,400 rows (ncu,
                     # profiles/k_decode_fast_kv_dense_link.md): every launch reads as many
                     "traffic": 310.93e6,
                     "traffic_is": "host-link (sysmem) read bytes of one launch from ncu "
                                   "(1.002 x its stored bytes)",
                     "kernel": "k_decode_fast<true, mode, big> (ibp_gather_decompress, 8 KB rows)"},
        "gpu_launches": 2 * L * args.steps,
        "clocks": clk.summary(),
        "decode_steps": decode,
        "decode_projection": proj,
        "cpu_baseline": leg,
        "attention_layout": {"value": round(att_gbs, 3), "unit": "GB/s", "steps": asteps,
                             "frac": round(att_gbs / roof, 4), "parity_layer0_ok": att_ok,
                             "note": "the same 64 gathers per step written as [20, 32, 1920, "
                                     "128] fp16 per layer and K|V (ibp_gather_decompress_split)"},
    }
    for st in stores:
        ibp.ibp_store_destroy(st)
    return res


def kv_decode_projection(torch, ibp, dev, stream, sp, seed=0, reps=50, tokens=20):
    """A decode step's K (or V) projection of one layer, OPT-6.7B shape: the
    20 new tokens' hidden states [20, 4096] fp16 times a 4096 x 4096 fp16
    weight (+ bias), each output row (one token's K: 8 KB) compressed into
    its host slot.  Fused (ibp_project_compress: tensor-core GEMM with the
    compressor in its epilogue) against the unfused pair (cuBLAS through
    torch, then ibp_compress).  The store's Mask/Bitval comes from the
    prompt's 20 x 1920 projected rows; weight rows carry per-channel
    log-normal scales with 2 % outlier channels x20, so the projected K/V
    follow the KV workload's recipe (N(0, 1) times per-channel scales).
    Parity: the fused slots, stored sizes and raw bits equal ibp_compress of
    the fused Y, and the oracle's compression of 20 rows equals both."""
    from oracle import ref_c
    B, P, T, CH = tokens, 1920, 2048, 4096
    R, C = CH * 2, 256
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 7 + 11)
    scale = torch.exp(0.5 * torch.randn(CH, generator=g, device=dev))
    scale[torch.randperm(CH, generator=g, device=dev)[:int(round(0.02 * CH))]] *= 20.0
    w = (torch.randn((CH, CH), generator=g, device=dev) * (scale[:, None] / CH ** 0.5)).half()
    bias = (torch.randn(CH, generator=g, device=dev) * 0.05 * scale).half()
    rows = 20 * T  # 20 sequences of 2048 token slots
    st = ibp.ibp_store_create(R, C, rows, R)
    # the prompt: 20 sequences x 1920 tokens whatever the decode batch
    xp = torch.randn((20 * P, CH), generator=g, device=dev).half()
    yp = torch.nn.functional.linear(xp, w, bias)
    pid = torch.from_numpy((np.arange(20)[:, None] * T + np.arange(P)[None, :]).reshape(-1)).to(dev)
    ibp.ibp_build_meta(st, yp.view(torch.uint8), R, None, 20 * P, 95, 100)
    slots = torch.empty((rows, R), dtype=torch.uint8, pin_memory=True)
    slots2 = torch.empty((rows, R), dtype=torch.uint8, pin_memory=True)
    ibp.ibp_compress(st, slots, yp.view(torch.uint8), R, pid, 20 * P, None)
    del xp, yp
    x = torch.randn((B, CH), generator=g, device=dev).half()
    # token i goes to sequence i % 20, decode position i // 20 (distinct slots)
    sid = torch.from_numpy(((np.arange(B) % 20) * T + P + np.arange(B) // 20)
                           .astype(np.int64)).to(dev)
    y = torch.empty((B, CH), dtype=torch.float16, device=dev)
    stored = torch.empty(B, dtype=torch.int32, device=dev)
    stored2 = torch.empty(B, dtype=torch.int32, device=dev)
    wsb = ibp.project_workspace_bytes(B, R)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def fused():
        ibp.ibp_project_compress(st, x, B, CH, w, bias, 0, y, slots, sid, stored, ws, wsb, sp)

    def unfused():
        yu = torch.nn.functional.linear(x, w, bias)
        ibp.ibp_compress(st, slots2, yu, R, sid, B, stored2, sp)

    def timeit(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.zero_()  # the 32 MB weight comes from HBM, as in a decode step
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    with ClockSampler(dev.index) as clk:
        t_f = timeit(fused)
        t_u = timeit(unfused)
        t_g = timeit(lambda: torch.nn.functional.linear(x, w, bias))
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    # parity: the fused result against ibp_compress of the fused Y, and the oracle
    fused()
    ibp.ibp_compress(st, slots2, y, R, sid, B, stored2, sp)
    torch.cuda.synchronize()
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    sid_np = sid.cpu().numpy()
    st_f = stored.cpu().numpy().astype(np.uint32)
    st_u = stored2.cpu().numpy().astype(np.uint32)
    s1, s2 = slots.numpy(), slots2.numpy()
    same = bool(np.array_equal(st_f, st_u)) and all(
        np.array_equal(s1[i, :st_f[j]], s2[i, :st_f[j]]) for j, i in enumerate(sid_np))
    mask = np.zeros(R // 4, np.uint32)
    bitval = np.zeros(R // 4, np.uint32)
    ibp.ibp_meta_get(st, mask, bitval)
    yb = y.view(torch.uint8).cpu().numpy().reshape(B, R)
    ref_sl = np.zeros((B, R), np.uint8)
    ref_bm = np.zeros((B + 31) // 32, np.uint32)
    ref_st = ref_c.compress_batch(yb, C, mask, bitval, ref_sl, ref_bm)
    oracle_ok = bool(np.array_equal(ref_st, st_f)) and all(
        np.array_equal(s1[i, :ref_st[j]], ref_sl[j, :ref_st[j]]) for j, i in enumerate(sid_np))
    ibp.ibp_store_destroy(st)
    wbytes = CH * CH * 2 + B * CH * 2  # the weight, and X: the kernel's algorithmic reads
    hbm = measured_peaks()["hbm_gbs"]
    return {"tokens": B, "fused_us": round(t_f, 2), "unfused_us": round(t_u, 2),
            "gemm_us": round(t_g, 2),
            "roofline": {"bound": "hbm", "achieved": round(wbytes / t_f / 1e3, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(wbytes / t_f / 1e3 / hbm, 4),
                         # dram__bytes_read.sum of one 20-token launch of
                         # k_project_compress<4, 32> (profiles/
                         # k_project_compress_kv_decode.md); null at other sizes
                         "traffic": 33.82e6 if B == 20 else None,
                         "kernel": "k_project_compress + k_project_assemble (whole call)"},
            "fused_speedup": round(t_u / t_f, 3),
            "weight_gbs_fused": round(CH * CH * 2 / t_f / 1e3, 1),
            "ratio": round(float(st_f.sum()) / (B * R), 5),
            "parity_vs_unfused_ok": same, "parity_oracle_ok": oracle_ok,
            "clocks": clk.summary(),
            "note": "one (layer, K) projection of a decode step: 20 x 4096 fp16 times 4096 x "
                    "4096 (+ bias); fused ibp_project_compress vs cuBLAS (torch) + ibp_compress; "
                    "a step has 64 such calls (32 layers x K, V); L2 flushed before each"}


def run_project(args, rank, world, torch, dist):
    """The K/V projection with the compressor in its epilogue at several
    decode batch sizes (tokens per call: 20 is a decode step of the KV
    workload), fused against cuBLAS + ibp_compress; the value is the fused
    call's weight-streaming GB/s at 20 tokens."""
    from lossless_invariant_bit_gb300 import ibp

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    pts = [kv_decode_projection(torch, ibp, dev, stream, sp, seed=args.seed, tokens=m,
                                reps=max(10, min(args.steps, 50)))
           for m in (20, 160, 1280)]
    head = pts[0]
    return {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": head["weight_gbs_fused"], "unit": "GB/s (weight streamed)", "n_gpus": world,
        "steps": max(10, min(args.steps, 50)), "warmup": 5,
        "ms_per_step": round(head["fused_us"] / 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded torch generator: OPT-6.7B K projection shapes)",
        "config": {"workload": "K/V projection + compression, 4096 x 4096 fp16 weight, "
                               "tokens 20 / 160 / 1280 per call"},
        "points": pts, "gpu_launches": 2, "clocks": head["clocks"]}


def run_weights(args, rank, world, torch, dist):
    """bf16 weight offloading (the pages' LLM weight-offload stream): the
    weights of L transformer layers of OPT-6.7B shape (q, k, v, o: 4096 x 4096;
    fc1: 16384 x 4096; fc2: 4096 x 16384, all as rows of 4096 bf16 = 8 KB),
    N(0, 0.02^2), compressed into pinned host slots, one store per matrix,
    Mask/Bitval from a 1 % sample, chunk 256 B.  A step streams one layer's
    six matrices back to HBM (six ibp_decompress launches, 384 MB of weights),
    layers in turn."""
    from lossless_invariant_bit_gb300 import dist as ibpdist
    from lossless_invariant_bit_gb300 import ibp
    from lossless_invariant_bit_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    args = argparse.Namespace(**vars(args))
    args.steps = min(args.steps, 64)
    L, R, C = args.weight_layers, 8192, 256
    mats = [4096, 4096, 4096, 4096, 16384, 16384]  # rows per matrix
    layer_rows = sum(mats)
    t0 = time.time()
    g = torch.Generator(device=dev)
    stores, slots, stored_tot = [], [], 0
    check, lengths = [], []
    for layer in range(L):
        for m, nr in enumerate(mats):
            g.manual_seed(args.seed * 1000003 + layer * 8 + m)
            w = (torch.randn((nr, 4096), generator=g, device=dev) * 0.02).to(torch.bfloat16)
            wb = w.view(torch.uint8)
            st = ibp.ibp_store_create(R, C, nr, 0)
            sample = torch.from_numpy(wl.sample_ids(nr, 10, seed=layer * 8 + m)).to(dev)
            ibp.ibp_build_meta(st, wb, R, sample, len(sample), 95, 100)
            sl = torch.empty((nr, R), dtype=torch.uint8, pin_memory=True)
            stored = torch.empty(nr, dtype=torch.int32, device=dev)
            ibp.ibp_compress(st, sl, wb, R, None, nr, stored)
            stored_tot += int(stored.sum().item())
            ibp.ibp_store_set_lengths(st, stored)  # whole streams in one fetch
            lengths.append(stored)
            if layer == 0:
                check.append(wb.clone())
            stores.append(st)
            slots.append(sl)
            del w, wb
    torch.cuda.synchronize()
    log("weight store ready in %.1fs" % (time.time() - t0))
    ratio = stored_tot / (L * layer_rows * R)
    out = torch.empty((layer_rows, R), dtype=torch.uint8, device=dev)
    offs = np.cumsum([0] + mats)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def step(b):
        layer = b % L
        for m, nr in enumerate(mats):
            k = layer * len(mats) + m
            ibp.ibp_decompress(stores[k], out[offs[m]:offs[m + 1]], slots[k], None, nr, sp)

    for b in range(args.warmup):
        step(b)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    evs = []
    with ClockSampler(dev.index) as clk:
        for b in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step(args.warmup + b)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    for st in stores:
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    times = [a.elapsed_time(c) / 1e3 for a, c in evs]
    t_total = ibpdist.max_over_ranks(sum(times), dist, dev)
    value = layer_rows * R * args.steps * world / t_total / 1e9
    step(0)
    torch.cuda.synchronize()
    parity_ok = all(bool(torch.equal(out[offs[m]:offs[m + 1]], check[m])) for m in range(len(mats)))
    link = _link_probe(torch, ibp, slots[4], stream, sp, dev)
    roof = min(measured_peaks()["hbm_gbs"], link / ratio)
    res = {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_total / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded torch generator on the GPU: bf16 N(0, 0.02^2) weights)",
        "config": {"workload": "bf16 weight offload: %d layers of OPT-6.7B shape (q, k, v, o, "
                               "fc1, fc2; 384 MB per layer) in pinned host slots, chunk 256 B, "
                               "1%% sample, T=0.95; one step = one layer's 6 matrices "
                               "decompressed into HBM" % L,
                   "row_bytes": R, "chunk_bytes": C, "launches_per_step": len(mats),
                   "l2": "flushed between steps (256 MB write, outside the timed events)"},
        "ratio": round(ratio, 5), "space_saving": round(1 - ratio, 4), "link_gbs": round(link, 2),
        "parity_layer0_ok": parity_ok,
        "roofline": {"bound": "link", "achieved": round(value / world, 2), "peak": round(roof, 2),
                     "unit": "GB/s", "frac": round(value / world / roof, 4), "traffic": None,
                     "kernel": "k_decode_fast<false, mode, big> (ibp_decompress, 8 KB rows)"},
        "gpu_launches": len(mats) * args.steps,
        "clocks": clk.summary(),
    }
    for st in stores:
        ibp.ibp_store_destroy(st)
    return res


def run_large(args, rank, world, torch, dist):
    """Gathers from a host store larger than the GPU's reach into host memory:
    sparse-GNN rows (128 fp32, 1.0 w.p. 0.01) generated on the GPU in chunks
    (seeded torch generator per chunk), compressed into pinned host slots of
    --large-rows rows (50M rows = 25.6 GB by default); 1 % sample of the first
    chunk, T = 0.95, chunk 1 KB.  A step gathers 200,000 uniform ids, by the
    plain gather and by the ordered gather (ids bucketed by address first)."""
    from lossless_invariant_bit_gb300 import ibp
    from lossless_invariant_bit_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    N, R, C, n = args.large_rows, 512, 1024, args.batch
    chunk = 1 << 20
    t0 = time.time()
    st = ibp.ibp_store_create(R, C, N, 0)
    slot = ibp.ibp_store_get_info(st).slot_bytes
    slots = torch.empty((N, slot), dtype=torch.uint8, pin_memory=True)
    g = torch.Generator(device=dev)

    def gen(c0, cnt):
        g.manual_seed(args.seed * 1000003 + c0 // chunk)
        return (torch.rand((cnt, 128), generator=g, device=dev) < 0.01).to(torch.float32)

    first = gen(0, min(chunk, N)).view(torch.uint8)
    sample = torch.from_numpy(wl.sample_ids(first.shape[0], 10, seed=args.seed)).to(dev)
    ibp.ibp_build_meta(st, first, R, sample, len(sample), 95, 100)
    torch.cuda.synchronize()
    stored_all = torch.empty(N, dtype=torch.int32, device=dev)
    for c0 in range(0, N, chunk):
        cnt = min(chunk, N - c0)
        rows = gen(c0, cnt).view(torch.uint8)
        sids = torch.arange(c0, c0 + cnt, dtype=torch.int64, device=dev)
        ibp.ibp_compress(st, slots, rows, R, sids, cnt, stored_all[c0:c0 + cnt])
    torch.cuda.synchronize()
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    log("large store: %d rows (%.1f GB of host slots) in %.1fs" % (N, N * slot / 1e9,
                                                                  time.time() - t0))
    pool = 8
    ids = [torch.from_numpy(wl.uniform_ids(n, N, seed=args.seed, batch=b)).to(dev)
           for b in range(pool)]
    stored_np = stored_all.cpu().numpy().astype(np.int64)
    ratio = statistics.mean(float(stored_np[x.cpu().numpy()].sum()) / (n * R) for x in ids)
    out = torch.empty((n, R), dtype=torch.uint8, device=dev)
    out2 = torch.empty((n, R), dtype=torch.uint8, device=dev)
    ws = torch.empty(ibp.order_workspace_bytes(n), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    steps = max(3, min(args.steps, 50))

    def timed(fn):
        for b in range(3):
            fn(b)
        evs = []
        for b in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(b)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(c) / 1e3 for a, c in evs)

    with ClockSampler(dev.index) as clk:
        t_plain = timed(lambda b: ibp.ibp_gather_decompress(st, out, slots, None, ids[b % pool],
                                                             n, sp))
        t_ord = timed(lambda b: ibp.ibp_gather_decompress_ordered(st, out2, R, slots, None,
                                                                   ids[b % pool], n, ws,
                                                                   ws.numel(), sp))
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    last = (2 + steps) % pool
    ibp.ibp_gather_decompress(st, out, slots, None, ids[last], n, sp)
    ibp.ibp_gather_decompress_ordered(st, out2, R, slots, None, ids[last], n, ws, ws.numel(), sp)
    torch.cuda.synchronize()
    same = bool(torch.equal(out, out2))
    # sampled rows against the generator: chunk by chunk
    pick = np.random.default_rng(3).choice(n, 256, replace=False)
    idl = ids[last].cpu().numpy()
    ok = True
    for k in pick[:32]:
        r = int(idl[k])
        c0 = (r // chunk) * chunk
        row = gen(c0, min(chunk, N - c0))[r - c0].view(torch.uint8)
        ok &= bool(torch.equal(out2[int(k)], row))
    link = _link_probe(torch, ibp, slots[: min(N, 1 << 21)], stream, sp, dev)
    roof = min(measured_peaks()["hbm_gbs"], link / ratio)
    v_plain, v_ord = n * R / t_plain / 1e9, n * R / t_ord / 1e9
    ibp.ibp_store_destroy(st)
    return {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": round(v_ord, 3), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": 3, "ms_per_step": round(t_ord * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded torch generator on the GPU: sparse GNN features)",
        "config": {"workload": "large host store: %d x 128 fp32 sparse rows (%.1f GB of pinned "
                               "host slots), chunk 1 KB, T=0.95; gathers of %d uniform ids, "
                               "ordered" % (N, N * slot / 1e9, n),
                   "l2": "flushed between steps (256 MB write, outside the timed events)"},
        "ratio": round(ratio, 5), "link_gbs": round(link, 2),
        "plain_gather": {"value": round(v_plain, 3), "frac": round(v_plain / roof, 4)},
        "ordered_gather": {"value": round(v_ord, 3), "frac": round(v_ord / roof, 4)},
        "ordered_equals_plain": same, "parity_sampled_rows_ok": ok,
        "roofline": {"bound": "link", "achieved": round(v_ord, 2), "peak": round(roof, 2),
                     "unit": "GB/s", "frac": round(v_ord / roof, 4), "traffic": None,
                     "kernel": "k_decode_fast<true, mode, small> (ordered gather)"},
        "gpu_launches": 4 * steps, "clocks": clk.summary(),
    }


def run_dlrm(args, rank, world, torch, dist):
    """DLRM embedding lookup: 26 tables x 1,000,000 rows of fp32 ~ N(0, 0.01^2)
    (dim 128/256/512: 512 B - 2 KB rows) compressed into pinned host slots
    (13.3 GB at dim 128), one Mask/Bitval per table from a 1 % sample, T = 0.95,
    chunk 1 KB.  A step is one batch of 8192 lookups, one Zipf(1.05) index per
    table (through a seeded permutation), gather-decompressed into a dense
    [8192, 26, dim] HBM tensor."""
    from lossless_invariant_bit_gb300 import dist as ibpdist
    from lossless_invariant_bit_gb300 import ibp
    from lossless_invariant_bit_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    Tn, N, dim, B, C = 26, args.dlrm_rows, args.dlrm_dim, 8192, 1024
    R = dim * 4
    t0 = time.time()
    stores, slots, tables_ok = [], [], []
    g = torch.Generator(device=dev)
    stored_sum = []
    check_rows = []
    lengths = []  # each table's stored sizes, attached to its store (length table)
    batches = [np.stack([wl.zipf_ids(B, N, table=t, seed=args.seed * 1000 + bb)
                         for t in range(Tn)], axis=1) for bb in range(min(args.pool, 4))]
    for t in range(Tn):
        g.manual_seed(args.seed * 7919 + t)
        x = (torch.randn((N, dim), generator=g, device=dev) * 0.01).view(torch.uint8)
        st = ibp.ibp_store_create(R, C, N, R)
        sample = torch.from_numpy(wl.sample_ids(N, 10, seed=args.seed + t)).to(dev)
        ibp.ibp_build_meta(st, x, R, sample, sample.numel(), 95, 100)
        sl = torch.empty((N, R), dtype=torch.uint8, pin_memory=True)
        stored = torch.empty(N, dtype=torch.int32, device=dev)
        ibp.ibp_compress(st, sl, x, R, None, N, stored)
        ibp.ibp_store_set_lengths(st, stored)
        lengths.append(stored)
        stored_sum.append(stored.to(torch.int64).cpu().numpy())
        # the rows the last batch looks up in this table, for the parity check
        check_rows.append(x[torch.from_numpy(batches[-1][:, t]).to(dev)].cpu())
        stores.append(st)
        slots.append(sl)
        del x
    torch.cuda.synchronize()
    log("DLRM store ready in %.1fs" % (time.time() - t0))
    ids_dev = [[torch.from_numpy(np.ascontiguousarray(bt[:, t])).to(dev) for t in range(Tn)]
               for bt in batches]
    out = torch.empty((B, Tn, R), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    pool = len(batches)

    def step(b):
        ids = ids_dev[b % pool]
        for t in range(Tn):
            ibp.ibp_gather_decompress_strided(stores[t], out[:, t], Tn * R, slots[t], None,
                                              ids[t], B, sp)

    for b in range(args.warmup):
        step(b)
    step(pool - 1)
    torch.cuda.synchronize()
    parity_ok = all(torch.equal(out[:, t].cpu(), check_rows[t]) for t in range(Tn))
    evs = []
    with ClockSampler(dev.index) as clk:
        for b in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step(b)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
    for st in stores:
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    per_store_times = [a.elapsed_time(c) / 1e3 for a, c in evs]
    per_store_gbs = B * Tn * R * len(per_store_times) / sum(per_store_times) / 1e9
    # the uncompressed transfer of the same lookups over the same host memory:
    # 26 raw gathers of R bytes from the same slot addresses (the slots are R
    # bytes apart), the review's Table 1 baseline for this workload
    raw_out = torch.empty((Tn, B, R), dtype=torch.uint8, device=dev)

    def step_raw(b):
        ids = ids_dev[b % pool]
        for t in range(Tn):
            ibp.ibp_gather_copy(raw_out[t], slots[t], R, R, ids[t], B, N, sp)
    for b in range(args.warmup):
        step_raw(b)
    rev = []
    for b in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step_raw(b)
        e1.record(stream)
        rev.append((e0, e1))
    torch.cuda.synchronize()
    raw_gbs = B * Tn * R * len(rev) / sum(a.elapsed_time(c) / 1e3 for a, c in rev) / 1e9
    del raw_out

    # the same batches through one fused launch over all 26 tables
    grp = ibp.ibp_group_create(stores, slots)
    ids2d = [torch.from_numpy(np.ascontiguousarray(bt)).to(dev) for bt in batches]

    def step_fused(b):
        ibp.ibp_group_gather_decompress(grp, out, Tn * R, ids2d[b % pool], B, sp)

    out.zero_()
    for b in range(args.warmup):
        step_fused(b)
    step_fused(pool - 1)
    torch.cuda.synchronize()
    fused_ok = all(torch.equal(out[:, t].cpu(), check_rows[t]) for t in range(Tn))
    evs = []
    with ClockSampler(dev.index) as clk:
        for b in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step_fused(b)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
    for st in stores:
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    times = [a.elapsed_time(c) / 1e3 for a, c in evs]
    # the same fused gather in address order (items bucketed by table and
    # region first: the tables together outgrow the GPU's reach into host memory)
    ws = torch.empty(ibp.order_workspace_bytes(B * Tn), dtype=torch.uint8, device=dev)
    out_o = torch.empty_like(out)

    def step_ordered(b):
        ibp.ibp_group_gather_decompress_ordered(grp, out_o, Tn * R, ids2d[b % pool], B, ws,
                                                ws.numel(), sp)

    for b in range(args.warmup):
        step_ordered(b)
    step_fused(pool - 1)
    step_ordered(pool - 1)
    torch.cuda.synchronize()
    ordered_same = bool(torch.equal(out, out_o))
    oev = []
    with ClockSampler(dev.index) as clk_o:
        for b in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step_ordered(b)
            e1.record(stream)
            oev.append((e0, e1))
        torch.cuda.synchronize()
    for st in stores:
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    # the same ordered gathers with each batch's plan made one step ahead: a
    # step gathers batch b (planned during the step before) while a second
    # stream plans batch b + 1; the step ends when both are done, and the plan
    # starts no earlier than the step (two workspaces in turn)
    wsb = ibp.order_workspace_bytes(B * Tn)
    pws = [torch.empty(wsb, dtype=torch.uint8, device=dev) for _ in range(2)]
    out_p = torch.empty_like(out)
    ps = torch.cuda.Stream(device=dev)
    planned = [torch.cuda.Event(), torch.cuda.Event()]
    gathered = [torch.cuda.Event(), torch.cuda.Event()]
    ps.wait_stream(stream)
    ibp.ibp_group_order_plan(grp, ids2d[0], B, pws[0], wsb, ps.cuda_stream)
    planned[0].record(ps)

    def step_piped(b, start=None):
        k = b % 2
        stream.wait_event(planned[k])
        ibp.ibp_group_gather_decompress_planned(grp, out_p, Tn * R, ids2d[b % pool], B, pws[k],
                                                wsb, sp)
        gathered[k].record(stream)
        if start is not None:
            ps.wait_event(start)
        ps.wait_event(gathered[1 - k])  # the previous step's gather read that workspace
        ibp.ibp_group_order_plan(grp, ids2d[(b + 1) % pool], B, pws[1 - k], wsb, ps.cuda_stream)
        planned[1 - k].record(ps)
        stream.wait_event(planned[1 - k])

    for b in range(args.warmup):
        step_piped(b)
    torch.cuda.synchronize()
    pev = []
    with ClockSampler(dev.index) as clk_p:
        for b in range(args.warmup, args.warmup + args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step_piped(b, start=e0)
            e1.record(stream)
            pev.append((e0, e1))
        torch.cuda.synchronize()
    for st in stores:
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    lastp = (args.warmup + args.steps - 1) % pool
    step_ordered(lastp)
    torch.cuda.synchronize()
    piped_same = bool(torch.equal(out_p, out_o))
    ptimes = [a.elapsed_time(c) / 1e3 for a, c in pev]
    # the step's parts timed apart (each with the L2 flushed before it): the
    # planned gather alone (its plan made once), the plan alone, and plan then
    # gather on one stream
    ibp.ibp_group_order_plan(grp, ids2d[0], B, pws[0], wsb, sp)
    parts = {"gather_alone_us": [], "plan_alone_us": [], "plan_then_gather_us": []}
    for name in parts:
        for b in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if name != "gather_alone_us":
                ibp.ibp_group_order_plan(grp, ids2d[b % pool], B, pws[0], wsb, sp)
            if name != "plan_alone_us":
                bb = 0 if name == "gather_alone_us" else b % pool
                ibp.ibp_group_gather_decompress_planned(grp, out_p, Tn * R, ids2d[bb], B, pws[0],
                                                        wsb, sp)
            e1.record(stream)
            parts[name].append((e0, e1))
    torch.cuda.synchronize()
    for st in stores:
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    parts = {k: round(statistics.mean(a.elapsed_time(c) * 1e3 for a, c in v), 1)
             for k, v in parts.items()}
    parts["pipelined_step_us"] = round(statistics.mean(ptimes) * 1e6, 1)
    # cpu_baseline leg: the oracle decodes sampled lookups of the last batch in
    # three tables from the same host slots; its rows must equal the GPU's and
    # the tables' rows, and its compression of those rows the stored bytes
    step_ordered(pool - 1)
    torch.cuda.synchronize()
    o_np = out_o.cpu().numpy()
    pick = np.random.default_rng(5).choice(B, 1024, replace=False)
    legs = []
    for t in (0, Tn // 2, Tn - 1):
        legs.append(oracle_leg(ibp, stores[t], slots[t], R, C, batches[pool - 1][pick, t],
                               o_np[pick, t], check_rows[t].numpy()[pick]))
    ibp.ibp_group_destroy(grp)
    otimes = [a.elapsed_time(c) / 1e3 for a, c in oev]
    plain_gbs = B * Tn * R * len(times) / sum(times) / 1e9
    ordered_gbs = B * Tn * R * len(otimes) / sum(otimes) / 1e9
    # the line's value: the pipelined steps (each gathers one batch and plans
    # the next one)
    t_total = ibpdist.max_over_ranks(sum(ptimes), dist, dev)
    value = B * Tn * R * args.steps * world / t_total / 1e9
    ratio = statistics.mean(
        sum(float(stored_sum[t][batches[b % pool][:, t]].sum()) for t in range(Tn)) / (B * Tn * R)
        for b in range(args.steps))
    # Zipf lookups repeat rows: a row fetched once can serve its repeats from the
    # GPU's caches, so the link need only carry each distinct row's stored bytes
    ratio_unique = statistics.mean(
        sum(float(stored_sum[t][np.unique(batches[b % pool][:, t])].sum()) for t in range(Tn))
        / (B * Tn * R) for b in range(min(args.steps, pool)))
    pbytes = (slots[0].numel() // 16) * 16
    probe = torch.empty(pbytes, dtype=torch.uint8, device=dev)
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ibp.ibp_link_copy(probe, slots[0], pbytes, sp)
        e1.record(stream)
        e1.synchronize()
        tt = e0.elapsed_time(e1) / 1e3
        best = tt if best is None else min(best, tt)
    link = pbytes / best / 1e9
    del probe
    roof = min(measured_peaks()["hbm_gbs"], link / ratio_unique)
    res = {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_total / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded torch generator on the GPU: N(0, 0.01^2) embedding tables)",
        "config": {"workload": "DLRM lookup: 26 tables x %d rows x dim %d fp32 in pinned host "
                               "slots, chunk 1 KB, 1%% sample, T=0.95; batch 8192 Zipf(1.05) ids "
                               "per table -> [8192, 26, %d], ordered fused gather with each "
                               "batch's plan made one step ahead on a second stream"
                               % (N, dim, dim),
                   "row_bytes": R, "launches_per_step": 6,
                   "length_tables": "each table's stored sizes attached (one fetch per row)",
                   "l2": "flushed between steps (256 MB write, outside the timed events)"},
        "ratio": round(ratio, 5), "ratio_distinct_rows": round(ratio_unique, 5),
        "link_gbs": round(link, 2),
        "parity_all_lookups_ok": bool(parity_ok and fused_ok and ordered_same and piped_same),
        "fused_unordered": {"value": round(plain_gbs, 3), "unit": "GB/s",
                            "frac": round(plain_gbs / roof, 4),
                            "note": "ibp_group_gather_decompress: items in batch order"},
        "ordered_one_call": {"value": round(ordered_gbs, 3), "unit": "GB/s",
                             "frac": round(ordered_gbs / roof, 4),
                             "ms_per_step": round(statistics.mean(otimes) * 1e3, 4),
                             "clocks": clk_o.summary(), "launches_per_step": 6,
                             "note": "ibp_group_gather_decompress_ordered: each batch planned "
                                     "and gathered in one call on one stream"},
        "pipelined_same_rows_as_one_call": piped_same,
        "pipeline_parts": parts,
        "per_store_launches": {"value": round(per_store_gbs, 3), "unit": "GB/s",
                               "launches_per_step": Tn,
                               "note": "26 ibp_gather_decompress_strided calls per batch"},
        "raw_gather_per_table": {"value": round(raw_gbs, 3), "unit": "GB/s",
                                 "speedup_of_ordered_ibp": round(value / world / raw_gbs, 3),
                                 "note": "26 uncompressed ibp_gather_copy calls per batch over "
                                         "the same slot addresses (R bytes per lookup)"},
        "roofline": {"bound": "link", "achieved": round(value / world, 2), "peak": round(roof, 2),
                     "unit": "GB/s", "frac": round(value / world / roof, 4),
                     # host-link read sectors of the first timed k_gather_group launch at this
                     # size (ncu, profiles/k_gather_group_dlrm.md); null at other sizes
                     "traffic": ({128: 48.39e6, 512: 191.52e6}.get(dim)
                                 if (N, B, Tn, args.seed) == (1_000_000, 8192, 26, 0) else None),
                     "traffic_is": "host-link (sysmem) read bytes of one k_gather_group launch "
                                   "from ncu",
                     "peak_is": "min(HBM, link / stored bytes of the batch's distinct rows per "
                                "delivered byte): repeats of a row can come from the GPU's caches",
                     "kernel": "k_gather_group, planned (ibp_group_gather_decompress_planned, "
                               "leaving each SM room for a grouping CTA; the next batch's plan: "
                               "three bucketing kernels, the grouping and share kernels, on a "
                               "second stream)"},
        "gpu_launches": 6 * args.steps,
        "clocks": clk_p.summary(),
        "cpu_baseline": {
            "value": round(len(legs) * 1024 * R / sum(len(pick) * R / (l["value"] * 1e9)
                                                       for l in legs) / 1e9, 4),
            "unit": "GB/s", "cores": legs[0]["cores"], "kind": "oracle",
            "sample": "1024 lookups of the last batch in tables 0, %d and %d decoded by the "
                      "oracle C decoder from the same host slots" % (Tn // 2, Tn - 1),
            "parity_oracle_ok": all(l["parity_oracle_ok"] for l in legs)},
    }
    for st in stores:
        ibp.ibp_store_set_lengths(st, None)
        ibp.ibp_store_destroy(st)
    del lengths
    return res


def line_bytes(stored: np.ndarray) -> np.ndarray:
    """Link bytes of reading `stored` bytes from a 128-byte boundary: whole
    lines, then a tail that costs 32, 64 or 128 bytes (measured by the
    transfers workload's read_granularity)."""
    full, r = np.divmod(np.asarray(stored, np.int64), 128)
    tail = np.select([r == 0, r <= 32, r <= 64], [0, 32, 64], 128)
    return full * 128 + tail


def sector_bytes(start: np.ndarray, stored: np.ndarray) -> np.ndarray:
    """32-byte sectors touched by reading `stored` bytes from byte `start`."""
    start = np.asarray(start, np.int64)
    end = start + np.asarray(stored, np.int64)
    return (-(-end // 32) - start // 32) * 32


def dense_packed_host(torch, ibp, st, slots, stored, NR, R, ids_np, ids_dev, out, rb, timed,
                      link, raw_gbs, sp, dev):
    """The same store packed into pinned host memory: each row's stored bytes
    at a 16-byte offset (the packed layout of the HBM cache, System
    Integration), gathered through the offsets form of ibp_gather_decompress.
    Against the slot store (every stream from a 128-byte boundary) it trades
    line-aligned starts for no padding; the sector count says what the link
    would carry if it moved 32-byte sectors."""
    offs = torch.empty(NR + 1, dtype=torch.int64, device=dev)
    ibp.ibp_pack(st, None, offs, slots, stored, NR, sp)
    total = int(offs[NR].item())
    packed_dev = torch.empty(total, dtype=torch.uint8, device=dev)
    ibp.ibp_pack(st, packed_dev, offs, slots, stored, NR, sp)
    packed = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    packed.copy_(packed_dev)
    del packed_dev
    torch.cuda.synchronize()
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    gbs = timed(lambda b: ibp.ibp_gather_decompress(st, out, packed, offs, ids_dev[b % len(ids_np)],
                                                    len(ids_np[b % len(ids_np)]), sp))
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    x = ids_np[-1]
    ibp.ibp_gather_decompress(st, out, packed, offs, ids_dev[-1], len(x), sp)
    torch.cuda.synchronize()
    assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
    ok = bool(np.array_equal(out[:len(x)].cpu().numpy(), rb[x]))
    st_np = stored.cpu().numpy().astype(np.int64)
    off_np = offs[:NR].cpu().numpy()
    nb = sum(len(i) for i in ids_np) * R
    sec_packed = sum(float(sector_bytes(off_np[i], st_np[i]).sum()) for i in ids_np) / nb
    sec_slots = sum(float(sector_bytes(0, st_np[i]).sum()) for i in ids_np) / nb
    line_slots = sum(float(line_bytes(st_np[i]).sum()) for i in ids_np) / nb
    log("dense C=1024, packed host store (%.0f MB): %.1f GB/s  %.3fx raw; sectors per row byte "
        "%.4f packed / %.4f slots; link lines per row byte (slots) %.4f"
        % (total / 1e6, gbs, gbs / raw_gbs, sec_packed, sec_slots, line_slots))
    del packed
    return {"chunk_bytes": 1024, "store_bytes": total, "gbs": round(gbs, 2),
            "speedup_vs_raw_gather": round(gbs / raw_gbs, 3),
            "frac_of_link_over_sector_ratio": round(gbs / (link / sec_packed), 4),
            "sector_bytes_per_row_byte": round(sec_packed, 5),
            "slot_store_sector_bytes_per_row_byte": round(sec_slots, 5),
            "slot_store_line_bytes_per_row_byte": round(line_slots, 5),
            "parity_batch_ok": ok}


def run_dense(args, rank, world, torch, dist):
    """Dense GNN (the pages' Table 1 dense row): 2,000,000 x 128 fp32 features
    ~ N(0, 0.1^2) in pinned host slots (1 GB), Mask/Bitval from a 1 % sample at
    T = 0.95, chunk 256 B, 1 KB and 4 KB (1 KB and 4 KB give identical streams:
    one chunk per 512-byte row).  A step gathers one two-hop mini-batch, the
    sorted unique union of 1024 seeds, 15 neighbours each and 10 of each of
    those (uniform random graph).  Per chunk size: ratio, delivered GB/s, its
    fraction of link / ratio, and the speedup over the uncompressed gather of
    the same ids; the value is the 1 KB point."""
    from lossless_invariant_bit_gb300 import dist as ibpdist
    from lossless_invariant_bit_gb300 import ibp
    from lossless_invariant_bit_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    hbm = measured_peaks()["hbm_gbs"]
    NR, R = args.rows, 512
    steps, warm = max(3, min(args.steps, 200)), max(3, min(args.warmup, 10))
    rows = np.empty((NR, 128), np.float32)
    wl.dense_gnn_rows(NR, 128, seed=args.seed, out=rows)
    rb = rows.view(np.uint8)
    d_rows = torch.from_numpy(rb).to(dev)
    raw_host = torch.empty((NR, R), dtype=torch.uint8, pin_memory=True)
    raw_host.copy_(torch.from_numpy(rb))
    slots = torch.empty((NR, R), dtype=torch.uint8, pin_memory=True)
    link = _link_probe(torch, ibp, raw_host, stream, sp, dev)
    log("link probe: %.1f GB/s host->HBM" % link)
    sample = torch.from_numpy(wl.sample_ids(NR, 10, seed=args.seed)).to(dev)
    pool = 8
    ids_np = [wl.two_hop_ids(NR, seed=args.seed, batch=ibpdist.batch_seed(rank, b))
              for b in range(pool)]
    ids_dev = [torch.from_numpy(x).to(dev) for x in ids_np]
    nmax = max(len(x) for x in ids_np)
    out = torch.empty((nmax, R), dtype=torch.uint8, device=dev)
    stored = torch.empty(NR, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    launches = 0

    def timed(fn):
        nonlocal launches
        for b in range(warm):
            fn(b)
        evs = []
        for b in range(warm, warm + steps):
            flush.zero_()  # L2 flush, outside the timed events
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(b)
            e1.record(stream)
            evs.append((e0, e1, b % pool))
        torch.cuda.synchronize()
        launches += steps
        t = sum(a.elapsed_time(c) / 1e3 for a, c, _ in evs)
        return sum(len(ids_np[i]) for _, _, i in evs) * R / t / 1e9

    with ClockSampler(dev.index) as clk:
        raw_gbs = timed(lambda b: ibp.ibp_gather_copy(out, raw_host, R, R, ids_dev[b % pool],
                                                      len(ids_np[b % pool]), NR, sp))
        log("uncompressed gather: %.1f GB/s" % raw_gbs)
        points = []
        for C in (256, 1024, 4096):
            st = ibp.ibp_store_create(R, C, NR, 0)
            ibp.ibp_build_meta(st, d_rows, R, sample, len(sample), 95, 100)
            ibp.ibp_compress(st, slots, d_rows, R, None, NR, stored)
            torch.cuda.synchronize()
            assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
            st_np = stored.cpu().numpy().astype(np.int64)
            ratio = sum(float(st_np[x].sum()) for x in ids_np) / (sum(len(x) for x in ids_np) * R)
            gbs = timed(lambda b: ibp.ibp_gather_decompress(st, out, slots, None, ids_dev[b % pool],
                                                            len(ids_np[b % pool]), sp))
            assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
            last = (warm + steps - 1) % pool
            pick = np.random.default_rng(C).choice(len(ids_np[last]), 2000, replace=False)
            got_pick = out[torch.from_numpy(pick).to(dev)].cpu().numpy()
            ok = bool(np.array_equal(got_pick, rb[ids_np[last][pick]]))
            if C == 1024:  # cpu_baseline leg of the headline chunk size
                leg = oracle_leg(ibp, st, slots, R, C, ids_np[last][pick], got_pick,
                                 rb[ids_np[last][pick]],
                                 note="; 2000 ids of the last timed mini-batch")
            ideal = min(hbm, link / ratio)
            # what the link carries: whole 128-byte lines, a line's tail read
            # costing 32, 64 or 128 bytes (the transfers workload's
            # read_granularity); a 452-byte stream costs as much as a raw row
            line_ratio = sum(float(line_bytes(st_np[x]).sum()) for x in ids_np) / (
                sum(len(x) for x in ids_np) * R)
            gran = min(hbm, link / line_ratio)
            points.append({"chunk_bytes": C, "ratio": round(ratio, 5), "gbs": round(gbs, 2),
                           "roofline_peak": round(ideal, 2), "frac": round(gbs / ideal, 4),
                           "link_line_bytes_per_row_byte": round(line_ratio, 5),
                           "granular_peak": round(gran, 2),
                           "frac_of_granular_peak": round(gbs / gran, 4),
                           "speedup_vs_raw_gather": round(gbs / raw_gbs, 3),
                           "parity_sampled_rows_ok": ok})
            log("dense C=%d: ratio %.4f  %.1f GB/s  %.3f of link/ratio  %.3f of the line-granular "
                "ceiling  %.3fx raw" % (C, ratio, gbs, gbs / ideal, gbs / gran, gbs / raw_gbs))
            if C == 1024:
                packed_point = dense_packed_host(torch, ibp, st, slots, stored, NR, R, ids_np,
                                                 ids_dev, out, rb, timed, link, raw_gbs, sp, dev)
            ibp.ibp_store_destroy(st)
    head = next(p for p in points if p["chunk_bytes"] == 1024)
    n_avg = statistics.mean(len(x) for x in ids_np)
    return {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": head["gbs"], "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": round(n_avg * R / head["gbs"] / 1e6, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded numpy: dense GNN features N(0, 0.1^2); two-hop mini-batches "
                "on a uniform random graph)",
        "config": {"workload": "dense GNN gather-decompress: %d x 128 fp32 rows in pinned host "
                               "slots, 1%% sample, T=0.95; two-hop mini-batches of %.0f unique "
                               "ids on average; value is the 1 KB chunk point" % (NR, n_avg),
                   "l2": "flushed between steps (256 MB write, outside the timed events)"},
        "link_gbs": round(link, 2), "raw_gather_gbs": round(raw_gbs, 2),
        "roofline": {"bound": "link", "achieved": head["gbs"], "peak": head["roofline_peak"],
                     "unit": "GB/s", "frac": head["frac"],
                     # host-link read sectors of a 1 KB-chunk launch (ncu, 138,395 ids of a
                     # 400,000-row store: 15.03 sectors per id, profiles/
                     # k_decode_fast_kv_dense_link.md) scaled to this run's mean batch
                     "traffic": round(2080214 * 32 / 138395 * n_avg),
                     "traffic_is": "host-link (sysmem) read bytes per launch from ncu, scaled "
                                   "by the ids of a batch",
                     "kernel": "k_decode_fast<true, mode, small> (ibp_gather_decompress)"},
        "chunks": points,
        "packed_host_store": packed_point,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "cpu_baseline": leg,
    }


def _link_probe(torch, ibp, host, stream, sp, dev):
    """Best of 5 aligned zero-copy copies of a pinned host buffer into HBM, GB/s."""
    pbytes = (host.numel() // 16) * 16
    probe = torch.empty(pbytes, dtype=torch.uint8, device=dev)
    ibp.ibp_link_copy(probe, host, pbytes, sp)
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ibp.ibp_link_copy(probe, host, pbytes, sp)
        e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3
        best = t if best is None else min(best, t)
    del probe
    return pbytes / best / 1e9


def run_sweep(args, rank, world, torch, dist):
    """The pages' two sweeps, measured on this machine.

    Space saving (the review's Figure 7): rows whose words have exactly k
    invariant bits (k = 0, 4, ..., 28: space saving 0 to 87.5 %), either the k
    high bits of every word with one value (a uniform store: fp32 rows of one
    magnitude class) or k scattered positions per word with a per-word value
    (the general scatter network); rows of 4 KB at chunks of 256 B, 1 KB and
    4 KB, and rows of 1 KB at 256 B and 1 KB; 1 GB of pinned host slots, a step
    is one gather-decompress of 65,536 uniform ids.  Throughput is reported as
    a fraction of the ideal, link / ratio (decompression for free).

    Sampling (the review's sampling paragraph): the compression ratio of the
    sparse and dense GNN stores (2M x 128 fp32) with the Mask/Bitval built from
    1 %, 5 %, 10 % and all rows, at T = 0.95 and with the chunk-aware builder,
    and the builder's time."""
    from lossless_invariant_bit_gb300 import ibp
    from lossless_invariant_bit_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    hbm = measured_peaks()["hbm_gbs"]
    steps, warm = max(3, min(args.steps, 30)), 3
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    total = 1 << 30
    host = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    link = _link_probe(torch, ibp, host, stream, sp, dev)
    log("link probe: %.1f GB/s host->HBM" % link)
    n = 65536
    points, launches = [], 0
    gen = torch.Generator(device=dev)
    with ClockSampler(dev.index) as clk:
        for R, chunks in ((4096, (256, 1024, 4096)), (1024, (256, 1024))):
            N, W = total // R, R // 4
            slots = host.view(N, R)
            gen.manual_seed(args.seed * 1000003 + R)
            base = torch.randint(0, 256, (N, R), dtype=torch.uint8, device=dev,
                                 generator=gen).view(torch.int32)
            sample = torch.from_numpy(wl.sample_ids(N, 10, seed=args.seed)).to(dev)
            ids = [torch.from_numpy(wl.uniform_ids(n, N, seed=args.seed, batch=b)).to(dev)
                   for b in range(4)]
            out = torch.empty((n, R), dtype=torch.uint8, device=dev)
            stored = torch.empty(N, dtype=torch.int32, device=dev)
            pick = torch.from_numpy(np.random.default_rng(R).choice(n, 1000, replace=False)).to(dev)
            for scattered in (False, True):
                for k in range(0, 32, 4):
                    keep, const = wl.invariant_pattern(W, k, scattered, seed=args.seed)
                    rows = ((base & torch.from_numpy(keep.view(np.int32)).to(dev))
                            | torch.from_numpy(const.view(np.int32)).to(dev)).view(torch.uint8)
                    for C in chunks:
                        st = ibp.ibp_store_create(R, C, N, 0)
                        assert ibp.ibp_store_get_info(st).slot_bytes == R
                        ibp.ibp_build_meta(st, rows, R, sample, len(sample), 95, 100)
                        ibp.ibp_compress(st, slots, rows, R, None, N, stored)
                        torch.cuda.synchronize()
                        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
                        ratio = statistics.mean(
                            float(stored[x].sum().item()) / (n * R) for x in ids)
                        for b in range(warm):
                            ibp.ibp_gather_decompress(st, out, slots, None, ids[b % 4], n, sp)
                        evs = []
                        for b in range(steps):
                            flush.zero_()
                            e0 = torch.cuda.Event(enable_timing=True)
                            e1 = torch.cuda.Event(enable_timing=True)
                            e0.record(stream)
                            ibp.ibp_gather_decompress(st, out, slots, None, ids[b % 4], n, sp)
                            e1.record(stream)
                            evs.append((e0, e1))
                        torch.cuda.synchronize()
                        launches += steps
                        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
                        t = statistics.mean(a.elapsed_time(c) / 1e3 for a, c in evs)
                        last = ids[(steps - 1) % 4]
                        ok = bool(torch.equal(out[pick], rows.view(N, R)[last[pick]]))
                        gbs = n * R / t / 1e9
                        ideal = min(hbm, link / ratio)
                        points.append({"row_bytes": R, "chunk_bytes": C,
                                       "pattern": "scattered" if scattered else "high bits",
                                       "k": k, "saving": round(1 - ratio, 4),
                                       "ratio": round(ratio, 5), "gbs": round(gbs, 2),
                                       "ideal_gbs": round(ideal, 2),
                                       "frac": round(gbs / ideal, 4),
                                       "parity_sampled_rows_ok": ok})
                        log("R=%d C=%d %s k=%d: ratio %.3f  %.1f GB/s  %.3f of ideal" % (
                            R, C, points[-1]["pattern"], k, ratio, gbs, gbs / ideal))
                        ibp.ibp_store_destroy(st)
                    del rows
            del base, out, stored
            torch.cuda.empty_cache()

    # sampling sweep: ratio of the whole store against the share of rows analysed
    sampling = []
    cands = [(3, 4), (85, 100), (9, 10), (95, 100), (97, 100), (99, 100), (999, 1000), (1, 1)]
    for name, gen_rows in (("sparse GNN", wl.sparse_gnn_rows), ("dense GNN", wl.dense_gnn_rows)):
        NR, R, C = 2_000_000, 512, 1024
        rows_np = np.empty((NR, 128), np.float32)
        gen_rows(NR, 128, seed=args.seed, out=rows_np)
        d_rows = torch.from_numpy(rows_np.view(np.uint8)).to(dev)
        del rows_np
        slots_dev = torch.empty((NR, R), dtype=torch.uint8, device=dev)
        stored = torch.empty(NR, dtype=torch.int32, device=dev)
        chosen = torch.zeros(1, dtype=torch.int32, device=dev)
        for pm in (10, 50, 100, 1000):
            smp = None if pm == 1000 else torch.from_numpy(
                wl.sample_ids(NR, pm, seed=args.seed)).to(dev)
            ns = NR if smp is None else len(smp)
            st = ibp.ibp_store_create(R, C, NR, 0)
            ibp.ibp_build_meta(st, d_rows, R, smp, ns, 95, 100)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ibp.ibp_build_meta(st, d_rows, R, smp, ns, 95, 100)
            e1.record(stream)
            ibp.ibp_compress(st, slots_dev, d_rows, R, None, NR, stored)
            torch.cuda.synchronize()
            r95 = float(stored.sum().item()) / (NR * R)
            t_build = e0.elapsed_time(e1) / 1e3
            ibp.ibp_build_meta_tuned(st, d_rows, R, smp, ns, [c[0] for c in cands],
                                     [c[1] for c in cands], chosen, None, sp)
            ibp.ibp_compress(st, slots_dev, d_rows, R, None, NR, stored)
            torch.cuda.synchronize()
            assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
            rt = float(stored.sum().item()) / (NR * R)
            sampling.append({"workload": name, "sample_per_mille": pm, "sample_rows": ns,
                             "ratio_T0.95": round(r95, 5), "build_seconds": round(t_build, 6),
                             "ratio_tuned": round(rt, 5),
                             "tuned_T": "%d/%d" % cands[int(chosen.item())]})
            log("%s sample %d/1000: ratio %.4f (T=0.95), %.4f (tuned)" % (name, pm, r95, rt))
            ibp.ibp_store_destroy(st)
        del d_rows, slots_dev, stored
        torch.cuda.empty_cache()

    head = next(p for p in points if p["row_bytes"] == 4096 and p["chunk_bytes"] == 1024
                and p["pattern"] == "high bits" and p["k"] == 16)
    below = [p["frac"] for p in points if p["saving"] < 0.5]
    return {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": head["gbs"], "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": round(n * 4096 / head["gbs"] / 1e6, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded torch generator on the GPU for the saving sweep; seeded "
                "numpy GNN features for the sampling sweep)",
        "config": {"workload": "space-saving sweep: value is the 4 KB row, 1 KB chunk, 50 %% "
                               "saving point (high bits); gather of %d uniform ids from 1 GB "
                               "of pinned host slots" % n,
                   "l2": "flushed between steps (256 MB write, outside the timed events)"},
        "link_gbs": round(link, 2),
        "roofline": {"bound": "link", "achieved": head["gbs"], "peak": head["ideal_gbs"],
                     "unit": "GB/s", "frac": head["frac"], "traffic": None,
                     "kernel": "k_decode_fast<true, uniform, big> (4 KB rows, ibp_gather_decompress)"},
        "saving_sweep": points,
        "min_frac_below_50pct_saving": min(below),
        "sampling_sweep": sampling,
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }


def run_transfers(args, rank, world, torch, dist):
    """The review's Figure 5 on this machine: moving randomly chosen rows (tensors)
    from pinned host memory into HBM, by method and row size.  Rows are
    uncompressed; GB/s of rows delivered.  GPU aligned = ibp_gather_copy on
    128-byte aligned slots; GPU unaligned = the same kernel on a source shifted
    64 bytes off the line boundaries; CPU fine-grained = one cudaMemcpyAsync
    per row; CPU bulk = gather into a pinned staging buffer, then one copy.
    Timed with host wall clock to the stream's completion (the CPU methods do
    their work on the host)."""
    from lossless_invariant_bit_gb300 import ibp

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    total = 1 << 30
    res_sizes = {}
    for R in (128, 512, 2048, 8192):
        slot = ((R + 127) // 128) * 128
        N = total // slot
        host = torch.empty(N * slot + 128, dtype=torch.uint8, pin_memory=True)
        host.random_(0, 256)
        g = np.random.default_rng(R)
        n = min(100_000, N // 4)
        ids_np = g.integers(0, N - 1, size=n).astype(np.int64)
        ids_host = torch.from_numpy(ids_np).pin_memory()
        ids_dev = ids_host.to(dev)
        out = torch.empty((n, R), dtype=torch.uint8, device=dev)
        staging = torch.empty(n * R, dtype=torch.uint8, pin_memory=True)

        def wall(fn, reps):
            fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(reps):
                fn()
            torch.cuda.synchronize()
            return (time.perf_counter() - t0) / reps

        m = {}
        t = wall(lambda: ibp.ibp_gather_copy(out, host, slot, R, ids_dev, n, N, sp), 20)
        m["gpu_aligned"] = n * R / t / 1e9
        shifted = host.data_ptr() + 64
        t = wall(lambda: ibp.ibp_gather_copy(out, shifted, slot, R, ids_dev, n, N - 1, sp), 20)
        m["gpu_unaligned"] = n * R / t / 1e9
        nb = min(n, 20_000)
        t = wall(lambda: ibp.ibp_gather_copy_staged(out, host, slot, R, ids_host, nb, N, staging,
                                                     sp), 3)
        m["cpu_bulk"] = nb * R / t / 1e9
        nd = min(n, 5_000)
        t = wall(lambda: ibp.ibp_gather_copy_dma(out, host, slot, R, ids_host, nd, N, sp), 3)
        m["cpu_fine_grained"] = nd * R / t / 1e9
        # the aligned gather's output is checked against the host rows
        ibp.ibp_gather_copy(out, host, slot, R, ids_dev, n, N, sp)
        torch.cuda.synchronize()
        hv = host[:N * slot].view(N, slot)
        pick = torch.from_numpy(g.choice(n, 500, replace=False))
        ok = torch.equal(out.cpu()[pick], hv[torch.from_numpy(ids_np)[pick], :R])
        res_sizes[str(R)] = {k: round(v, 2) for k, v in m.items()}
        res_sizes[str(R)]["aligned_over_unaligned"] = round(m["gpu_aligned"] / m["gpu_unaligned"], 3)
        res_sizes[str(R)]["parity_ok"] = bool(ok)
        del host, staging, out
        torch.cuda.empty_cache()
    probe_src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    probe_dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    best = None
    for _ in range(5):
        ev[0].record(stream)
        ibp.ibp_link_copy(probe_dst, probe_src, 1 << 30, sp)
        ev[1].record(stream)
        ev[1].synchronize()
        tt = ev[0].elapsed_time(ev[1]) / 1e3
        best = tt if best is None else min(best, tt)
    # read granularity of the link: X bytes from the start of random 256-byte
    # slots (X = 16 .. 256); rows per microsecond show what each partly read
    # 128-byte line costs
    gran = []
    slot, N = 256, (1 << 30) // 256
    ng = 1 << 21
    ids_g = torch.from_numpy(np.random.default_rng(7).integers(0, N, size=ng).astype(np.int64)
                             ).to(dev)
    out_g = torch.empty(ng * slot, dtype=torch.uint8, device=dev)
    for X in range(16, 257, 16):
        for _ in range(3):
            ibp.ibp_gather_copy(out_g, probe_src, slot, X, ids_g, ng, N, sp)
        ts = []
        for _ in range(10):
            ev[0].record(stream)
            ibp.ibp_gather_copy(out_g, probe_src, slot, X, ids_g, ng, N, sp)
            ev[1].record(stream)
            ev[1].synchronize()
            ts.append(ev[0].elapsed_time(ev[1]) / 1e3)
        t = min(ts)
        gran.append({"row_bytes": X, "rows_per_us": round(ng / t / 1e6, 1),
                     "gbs": round(ng * X / t / 1e9, 2)})
    del out_g
    # the link's other directions, by the same copy kernel: HBM -> pinned host
    # (GPU stores over the link) and pinned host -> pinned host through the GPU
    # (reads and writes at once: the ceiling of an end-to-end call whose
    # inputs and outputs both live in host memory)
    host_dst = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dirs = {}
    for name, dst_, src_ in (("hbm_to_host", host_dst, probe_dst),
                             ("host_to_host_via_gpu", host_dst, probe_src)):
        bestd = None
        for _ in range(5):
            ev[0].record(stream)
            ibp.ibp_link_copy(dst_, src_, 1 << 30, sp)
            ev[1].record(stream)
            ev[1].synchronize()
            tt = ev[0].elapsed_time(ev[1]) / 1e3
            bestd = tt if bestd is None else min(bestd, tt)
        dirs[name + "_gbs"] = round((1 << 30) / bestd / 1e9, 2)
    del host_dst
    head = res_sizes["512"]["gpu_aligned"]
    return {
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": head, "unit": "GB/s", "n_gpus": 1, "steps": 20, "warmup": 1,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8", "data": "synthetic random bytes",
        "config": {"workload": "transfer methods (Figure 5 of the review): random rows of "
                               "128 B - 8 KB from 1 GB of pinned host memory into HBM"},
        "link_limit_gbs": round((1 << 30) / best / 1e9, 2),
        "by_row_bytes": res_sizes,
        "read_granularity": gran,
        "link_directions": dirs,
    }


def cpu_baseline(store, batches, ibp, seconds=1.5):
    """The oracle's decoder on the host cores over whole batches of this workload,
    until about `seconds` of wall time (x cores of CPU work) have been spent."""
    mask = np.zeros(store.R // 4, np.uint32)
    bitval = np.zeros(store.R // 4, np.uint32)
    ibp.ibp_meta_get(store.st, mask, bitval)
    bitmap = np.zeros((store.n_rows + 31) // 32, np.uint32)
    ibp.ibp_bitmap_get(store.st, bitmap)
    threads = len(os.sched_getaffinity(0))
    cpu_oracle_decode(store, batches[0][:1000], mask, bitval, bitmap, threads)  # warm
    rows, dt, k = 0, 0.0, 0
    while dt < seconds and k < len(batches):
        t0 = time.perf_counter()
        _, bad = cpu_oracle_decode(store, batches[k], mask, bitval, bitmap, threads)
        dt += time.perf_counter() - t0
        assert bad == 0
        rows += len(batches[k])
        k += 1
    # the same decoder on one core, over the first batch's first 20,000 ids
    t0 = time.perf_counter()
    cpu_oracle_decode(store, batches[0][:20000], mask, bitval, bitmap, 1)
    single = 20000 * store.R / (time.perf_counter() - t0) / 1e9
    return {"value": round(rows * store.R / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "single_core_gbs": round(single, 4),
            "kind": "oracle",
            "sample": "%d batches of %d ids of the same workload (%.1f s wall), oracle C "
                      "decoder, OpenMP over rows" % (k, len(batches[0]), dt)}


def oracle_leg(ibp, st, slots, R, C, ids, gpu_rows, raw_rows=None, threads=None,
               note=""):
    """The cpu_baseline leg of a sub-result: the oracle decodes rows `ids` of
    the same host slots on the host cores (timed), and its rows are compared
    byte for byte with the GPU's output for those ids (gpu_rows) and, when
    given, with the rows the store was compressed from (raw_rows), whose
    oracle compression must also equal the stored bytes in the slots."""
    from oracle import ref_c
    W = R // 4
    info = ibp.ibp_store_get_info(st)
    mask = np.zeros(W, np.uint32)
    bitval = np.zeros(W, np.uint32)
    ibp.ibp_meta_get(st, mask, bitval)
    bitmap = np.zeros((info.n_rows + 31) // 32, np.uint32)
    ibp.ibp_bitmap_get(st, bitmap)
    threads = threads or len(os.sched_getaffinity(0))
    slots_np = slots.numpy() if hasattr(slots, "numpy") else slots
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    t0 = time.perf_counter()
    out, bad = ref_c.decompress_batch(slots_np, bitmap, R, C, mask, bitval, ids=ids,
                                      slot_stride=int(info.slot_bytes), nthreads=threads)
    dt = time.perf_counter() - t0
    ok = bad == 0 and np.array_equal(out, gpu_rows)
    if raw_rows is not None:
        ok = ok and np.array_equal(out, raw_rows)
        # the oracle's own compression of the same rows: stored bytes and raw bits
        k = min(len(ids), 512)
        ref_sl = np.zeros((k, int(info.slot_bytes)), np.uint8)
        ref_bm = np.zeros((k + 31) // 32, np.uint32)
        ref_st = ref_c.compress_batch(np.ascontiguousarray(raw_rows[:k]), C, mask, bitval, ref_sl,
                                      ref_bm, nthreads=threads)
        sl2 = slots_np.reshape(info.n_rows, -1)
        for j in range(k):
            i = int(ids[j])
            ok = ok and bool(((bitmap[i >> 5] >> (i & 31)) & 1) == ((ref_bm[j >> 5] >> (j & 31)) & 1))
            ok = ok and np.array_equal(sl2[i, :ref_st[j]], ref_sl[j, :ref_st[j]])
    return {"value": round(len(ids) * R / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d rows of this workload decoded by the oracle C decoder (OpenMP over "
                      "rows, %.2f s)%s" % (len(ids), dt, note),
            "parity_oracle_ok": bool(ok)}


def free_host_cache(torch):
    """Return cached pinned host blocks and device blocks between workloads."""
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    if hasattr(torch._C, "_host_emptyCache"):
        torch._C._host_emptyCache()


def run_reference(args, rank, world, torch):
    """The oracle as it stands, on the host cores, same workload and metric."""
    from lossless_invariant_bit_gb300 import workloads as wl
    from oracle import ref_c

    n_rows, dim, R, C = 2_000_000, 128, 512, 1024
    rows = np.empty((n_rows, dim), np.float32)
    wl.sparse_gnn_rows(n_rows, dim, seed=args.seed, out=rows)
    rb = rows.view(np.uint8)
    sample = wl.sample_ids(n_rows, 10, seed=args.seed)
    threads = len(os.sched_getaffinity(0))
    mask, bitval = ref_c.build_meta(rb, 95, 100, sample_ids=sample)
    slot = 512
    slots = np.zeros((n_rows, slot), np.uint8)
    bitmap = np.zeros((n_rows + 31) // 32, np.uint32)
    ref_c.compress_batch(rb, C, mask, bitval, slots, bitmap, nthreads=threads)
    n = args.batch
    times = []
    pool = [wl.uniform_ids(n, n_rows, seed=args.seed, batch=b)
            for b in range(min(args.pool, args.warmup + args.steps))]
    for b in range(args.warmup + args.steps):
        ids = pool[b % len(pool)]
        t0 = time.perf_counter()
        _, bad = ref_c.decompress_batch(slots, bitmap, R, C, mask, bitval, ids=ids,
                                        slot_stride=slot, nthreads=threads)
        dt = time.perf_counter() - t0
        assert bad == 0
        if b >= args.warmup:
            times.append(dt)
    value = n * R * len(times) / sum(times) / 1e9
    return {
        "impl": "reference",
        "metric": "IBP decompressed GB/s delivered (host & HBM) and % of link/HBM roofline",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sum(times) / len(times) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded numpy: sparse GNN features)",
        "config": {"workload": "sparse GNN gather-decompress: 2,000,000 x 128 fp32 rows, "
                               "chunk 1 KB, 1% sample, T=0.95, batches of 200,000 uniform ids",
                   "source": "host memory (CPU oracle)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": "%d steps of %d ids, oracle C decoder" % (args.steps, n)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--rows", type=int, default=2_000_000)
    ap.add_argument("--pool", type=int, default=20, help="distinct id batches, cycled")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=200_000)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--workload", default="sparse",
                    choices=["sparse", "tiny", "kv", "dlrm", "transfers", "sweep", "weights",
                             "large", "dense", "project"])
    ap.add_argument("--dlrm-dim", type=int, default=128, choices=[128, 256, 512])
    ap.add_argument("--dlrm-rows", type=int, default=1_000_000)
    ap.add_argument("--kv-layers", type=int, default=32)
    ap.add_argument("--weight-layers", type=int, default=16)
    ap.add_argument("--large-rows", type=int, default=50_000_000)
    ap.add_argument("--replicas", type=int, default=128)
    ap.add_argument("--no-tuned", action="store_true",
                    help="skip the chunk-aware builder sub-result of the default workload")
    ap.add_argument("--no-cache-front", action="store_true",
                    help="skip the HBM cache-front sub-result of the default workload")
    ap.add_argument("--no-cache-path", action="store_true",
                    help="skip the HBM cache-path sub-result of the default workload")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the dense GNN, DLRM and KV sub-results of the default workload")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the CPU oracle: rank 0 alone runs it; other ranks exit without work
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world, torch)), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")

    from lossless_invariant_bit_gb300 import build as libbuild
    if rank == 0 or world == 1:
        libbuild.build()
    if dist:
        dist.barrier()
    run = {"tiny": run_tiny, "kv": run_kv, "dlrm": run_dlrm, "transfers": run_transfers,
           "sweep": run_sweep, "weights": run_weights,
           "large": run_large, "dense": run_dense,
           "project": run_project}.get(args.workload, run_ours)
    res = run(args, rank, world, torch, dist)
    if args.workload == "sparse" and not args.no_cache_path:
        # the HBM cache path of the same metric, reported beside the host path
        sub = argparse.Namespace(**vars(args))
        sub.steps, sub.warmup = min(args.steps, 200), max(3, min(args.warmup, 5))
        t = run_tiny(sub, rank, world, torch, dist)
        res["cache_path"] = {k: t[k] for k in ("value", "unit", "steps", "ms_per_step", "ratio",
                                               "parity_all_rows_ok", "single_batch_us", "roofline", "e2e",
                                               "clocks", "cpu_baseline")}
        res["cache_path"]["config"] = t["config"]["workload"]
    if args.workload == "sparse" and not args.no_configs and world > 1:
        # every rank would pin the full-size stores (53 GB for DLRM dim 512):
        # the scaling runs measure the headline alone
        res["configs"] = "dense GNN, DLRM and KV sub-results: run at one GPU only"
    if args.workload == "sparse" and not args.no_configs and world == 1:
        # the other workloads of the metric at their full sizes, each with its
        # own roofline, clock record and oracle leg (sub-results of this line)
        keep = ("value", "unit", "steps", "warmup", "ms_per_step", "ratio", "link_gbs",
                "roofline", "clocks", "cpu_baseline", "gpu_launches")
        subs = [("dense_gnn", run_dense, {}), ("dlrm_dim128", run_dlrm, {"dlrm_dim": 128}),
                ("dlrm_dim512", run_dlrm, {"dlrm_dim": 512}), ("kv_fetch", run_kv, {})]
        for key, fn, over in subs:
            free_host_cache(torch)
            sub = argparse.Namespace(**vars(args))
            sub.steps, sub.warmup = min(args.steps, 20), max(3, min(args.warmup, 5))
            for k_, v_ in over.items():
                setattr(sub, k_, v_)
            t0 = time.time()
            r = fn(sub, rank, world, torch, dist)
            d = {k_: r[k_] for k_ in keep if k_ in r}
            d["config"] = r["config"]
            for k_ in ("parity_all_lookups_ok", "parity_layer0_ok", "chunks", "fused_unordered",
                       "ordered_one_call", "pipelined_same_rows_as_one_call", "pipeline_parts",
                       "per_store_launches", "ratio_distinct_rows", "raw_gather_gbs",
                       "attention_layout", "decode_steps", "decode_projection",
                       "raw_gather_per_table", "packed_host_store"):
                if k_ in r:
                    d[k_] = r[k_]
            d["wall_s"] = round(time.time() - t0, 1)
            res[key] = d
            log("%s: %.1f GB/s (%.3f of its roofline) in %.0f s" % (
                key, r["value"], r["roofline"]["frac"], time.time() - t0))
        free_host_cache(torch)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
