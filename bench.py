"""Benchmark: paged decode attention over a tree-shaped KV cache on one GB300.

Default workload: ``long_context`` -- 64 q-heads / 8 kv-heads, head_dim 128,
bf16, block 16; 128 sequences of 8192 tokens plus 16 roots of 32768 tokens
each forked into 16 branches of 512 suffix tokens (6.98 GB of unique KV, far
larger than L2, so no L2 flush is needed between steps).  One step = one
``paged_decode_attn`` call: every kernel of the decode step (split-KV pass,
shared-prefix pass when tensor-core tiles exist, LSE merge) for all 384
branches.

Metric: unique-KV GB/s (distinct physical blocks read in the step x the valid
tokens of each x Hkv x d x 2 bytes x 2 for K and V, divided by the step
time); branch-queries/s is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline]

``--impl reference`` times the fp64 CPU oracle on the host cores (the only
reference implementation that exists for this path) on a bounded sample of
the same workload.  Under torchrun (N > 1) each rank runs an independent
replica of the workload (the path does not shard across GPUs): no collective
on the data path; the barrier and max-over-ranks timing stay.
"""

from __future__ import annotations

import os

# The oracle baseline parallelises over query rows with threads; keep BLAS to
# one thread per worker so "cores" is the number of threads really used.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import concurrent.futures as cf  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn: unique-KV GB/s vs HBM peak; branch-queries/sec"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--fused-steps", type=int, default=30)
    ap.add_argument("--offload-branches", type=int, default=32)
    ap.add_argument("--e4m3-steps", type=int, default=300)
    ap.add_argument("--profile-step", choices=["shared", "reread"],
                    help="run only `--steps` decode steps of --workload (plan "
                         "with its shared-prefix segments, or with every "
                         "branch re-reading its whole table) and exit: the "
                         "command ncu captures for the sharing figures")
    ap.add_argument("--per-config-steps", type=int, default=200,
                    help="steps for each of the other configurations (0: skip)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            low = line.lower()
            if low.startswith("model name") or low.startswith("cpu part"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def unique_kv_bytes(tables, seq_lens, Hkv, d, elem=2, record=0):
    """Distinct physical blocks read in the step, each weighted by the valid
    tokens in it, times Hkv * d * elem bytes * 2 (K and V); plus `record`
    bytes per distinct (block, kv-head) (the scale records of an e4m3
    pool)."""
    valid = {}
    for row, L in zip(tables, seq_lens):
        nblk = (int(L) + 15) // 16
        for j in range(nblk):
            n = min(16, int(L) - 16 * j)
            b = int(row[j])
            valid[b] = max(valid.get(b, 0), n)
    return (sum(valid.values()) * Hkv * d * elem * 2 +
            len(valid) * Hkv * record)


def plan_items(plan, info, which):
    """The work items of one kernel in a plan (int32 [n][8]: first branch,
    kv-head, first row, rows, block range, partial-row base, masked)."""
    off = 16 if which == "row" else 16 + 8 * info.n_row_items
    n = info.n_row_items if which == "row" else info.n_tile_items
    return plan[off:off + 8 * n].reshape(-1, 8)


def item_bytes(plan, info, Hkv, d, seq_lens, which, elem=2, record=0,
               segments_only=False):
    """Algorithmic KV bytes one launch of a kernel reads: for each of its work
    items, the valid tokens of its block range x 2 (K, V) x d x elem bytes,
    plus `record` bytes per block of the range (e4m3 scale records).  With
    segments_only, only the items over shared-prefix segments (masked == 0)
    count."""
    tot = blocks = 0
    for b0, g, row0, nr, lo, hi, pb, masked in plan_items(plan, info, which):
        if segments_only and masked:
            continue
        toks = (hi - lo) * 16
        if masked:
            toks = min(toks, int(seq_lens[b0]) - 16 * lo)
        tot += toks
        blocks += hi - lo
    return int(tot) * 2 * d * elem + int(blocks) * record


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_per_launch(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(f"{kernel}/{workload}")
    if not d:
        return None
    src = os.path.join(ROOT, "paged_kv_cache_attn_gb300", "csrc", d["source"])
    if not os.path.exists(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return d["dram_bytes_per_launch"] if sha == d["source_sha"] else None


def measured_sharing(workload):
    """Prefix bytes moved, re-read arm / shared arm, from the committed ncu
    summary (profiles/ncu_sharing.json) if it was taken on the current kernel
    sources; a workload is looked up under its own name or its quarter-size
    profiling case."""
    p = os.path.join(ROOT, "profiles", "ncu_sharing.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    for src, sha in d["sources"].items():
        f = os.path.join(ROOT, "paged_kv_cache_attn_gb300", "csrc", src)
        if (not os.path.exists(f) or
                hashlib.sha256(open(f, "rb").read()).hexdigest()[:16] != sha):
            return None
    e = d.get(workload) or d.get(workload + "_quarter")
    if not e:
        return None
    return {"case": workload if workload in d else workload + "_quarter",
            "branch_sharing_factor": e["branch_sharing_factor"],
            "prefix_bytes_to_sms_factor": e["prefix_tma_factor"],
            "prefix_l2_requests_factor": e["prefix_l2_tex_factor"],
            "prefix_dram_factor": e["prefix_dram_factor"],
            "source": "profiles/ncu_sharing.json"}


# ---- the oracle as the CPU baseline ----------------------------------------------

def prepare_sample(w, max_rows):
    """Pick up to max_rows batch rows (spread over the batch so every kind of
    branch is in it) and materialise their contiguous K/V and queries on the
    host.  Not timed: this is input preparation, not the oracle's work."""
    from oracle import replay as rp
    ref = rp.replay(w, with_data=False)
    nb = len(ref.decode_ids)
    q = w.queries(nb)
    rows = sorted(set(np.linspace(0, nb - 1, min(max_rows, nb)).astype(int)
                      .tolist()))
    sample = []
    for b in rows:
        k, v = ref.branch_kv(ref.decode_ids[b])
        sample.append((q[b], k[0], v[0]))
    return sample, nb


def oracle_unit(w, item, g):
    """The oracle on one (branch, kv-head): its G query heads against all of
    the branch's tokens.  Returns the KV bytes it read."""
    from oracle import attention as att
    qb, K, V = item
    G = w.Hq // w.Hkv
    att.attention(att.bf16_to_f64(qb[g * G:(g + 1) * G]),
                  att.bf16_to_f64(K[:, g]), att.bf16_to_f64(V[:, g]), w.scale)
    return K.shape[0] * w.d * 2 * 2


def run_units(w, sample, units, cores, ex):
    parts = [units[j::cores] for j in range(cores) if units[j::cores]]

    def part(us):
        return sum(oracle_unit(w, sample[i], g) for i, g in us)

    return sum(f.result() for f in [ex.submit(part, p) for p in parts])


def cpu_baseline(w, budget_s=12.0, threads=None):
    """Oracle throughput on host threads over a bounded sample of the batch:
    passes over the sampled (branch, kv-head) units until ~budget_s of wall
    time (at least one pass).  threads: how many (default: every core)."""
    sample, nb = prepare_sample(w, 24)
    units = [(i, g) for i in range(len(sample)) for g in range(w.Hkv)]
    cores = min(threads or host_cores(), len(units))
    done, byts, t0 = 0, 0, time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        while done < len(units) or time.perf_counter() - t0 < budget_s:
            chunk = [units[(done + i) % len(units)] for i in range(cores)]
            byts += run_units(w, sample, chunk, cores, ex)
            done += len(chunk)
    dt = time.perf_counter() - t0
    return {"value": round(byts / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{done} (branch, kv-head) oracle units ({done / len(units):.1f} "
                      f"passes over {len(sample)} of {nb} branches of {w.name}, "
                      f"{byts / 1e9:.1f} GB of KV read), fp64 numpy, "
                      f"{dt:.1f} s wall",
            "cpu": cpu_model()}


# ---- our arm ------------------------------------------------------------------------

KERNEL_NAMES = {"splitkv_mma": "splitkv_decode_kernel",
                "tile_tcgen05": "tile_decode_kernel"}


def tile_kernel_name(info):
    """The tcgen05 kernel(s) a plan's tile items run on."""
    n_wide = info.n_tile_wide_items
    names = (["tile_wide_kernel"] if n_wide else []) + \
        (["tile_decode_kernel"] if info.n_tile_items > n_wide else [])
    return "+".join(names)


def time_steps(bt, q, out, K, warmup, flush=None, before=None, after=None):
    """Time K decode steps after `warmup` untimed ones.  Returns (ms per step,
    per-kernel ms, per-step kernel events).

    Two passes of K steps each.  The first gives the step time: the steps
    run exactly as a caller runs them, with no per-kernel instrumentation
    (recording six events per step from Python slows short steps down).  The
    second has the library record, on the launching streams, events around
    each of its kernels; those windows give the per-kernel times and the
    roofline.  With `flush` (two device buffers, each larger than L2) the
    first is rewritten and the second read before each step -- the write
    evicts the step's KV from L2, the read then evicts the written lines, so
    that the step neither finds the previous one's KV in L2 nor pays for the
    flush's write-backs -- and each step is timed by its own pair of events.
    `before` / `after` (optional) run right before and right after the first
    pass, with the device synchronised on both sides (the ranks' barriers)."""
    import torch
    from paged_kv_cache_attn_gb300 import binding as B
    stream = torch.cuda.current_stream()
    for _ in range(max(warmup, 3)):
        bt.decode(q, out)
    torch.cuda.synchronize()
    code, detail = bt.device_status()
    if code:
        raise RuntimeError(f"device status {code} ({detail})")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)]
           for _ in range(K)]
    # torch creates the CUDA event behind an Event on its first record: do
    # that now, outside the timed region, so the library gets real handles.
    for row in evs:
        for e in row:
            e.record(stream)
    pairs = [(torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()

    def run(kernel_events):
        for i in range(K):
            if flush is not None:
                flush[0].add_(1)
                flush[1].sum()
                pairs[i][0].record(stream)
            if kernel_events:
                B.kv_set_launch_events(evs[i])
            bt.decode(q, out)
            if flush is not None:
                pairs[i][1].record(stream)
        B.kv_set_launch_events(None)

    if before is not None:
        before()
    torch.cuda.synchronize()
    start.record(stream)
    run(False)
    end.record(stream)
    torch.cuda.synchronize()
    if after is not None:
        after()
    if flush is None:
        ms = start.elapsed_time(end) / K
    else:
        ms = sum(a.elapsed_time(b) for a, b in pairs) / K
    run(True)
    torch.cuda.synchronize()
    per_kernel = {}
    for k, name in enumerate(["tile_tcgen05", "splitkv_mma", "lse_merge"]):
        if k == 0 and bt.info.n_tile_items == 0:
            continue
        if k == 1 and bt.info.n_row_items == 0:
            continue
        per_kernel[name] = sum(e[2 * k].elapsed_time(e[2 * k + 1])
                               for e in evs) / K
    code, detail = bt.device_status()
    if code:
        raise RuntimeError(f"device status {code} ({detail})")
    return ms, per_kernel, evs


def kernels_per_step(info):
    """This library's kernel launches in one step: the tile kernels (one for
    256-row items, one for 128-row items), the split-KV kernel, the merge."""
    n_wide = info.n_tile_wide_items
    return (int(n_wide > 0) + int(info.n_tile_items - n_wide > 0) +
            int(info.n_row_items > 0) + 1)


def kernel_roofline(bt, w, per_kernel, evs, peak, peak_kind):
    """Roofline of the dominant unit.  When the tile pass runs on its side
    stream beside the split pass, the two kernels share the GPU and each
    one's event window includes time spent queued behind the other: the unit
    is then the concurrent pair, its algorithmic bytes over the window from
    the first start to the last end (per step, averaged)."""
    alg_by = {k: item_bytes(bt.plan, bt.info, w.Hkv, w.d, bt.seq_lens,
                            "row" if k == "splitkv_mma" else "tile")
              for k in per_kernel if k != "lse_merge"}
    if len(alg_by) == 2:
        win = 0.0
        for e in evs:
            starts = [0.0, e[0].elapsed_time(e[2])]      # relative to tile start
            ends = [e[0].elapsed_time(e[1]), e[0].elapsed_time(e[3])]
            win += max(ends) - min(starts)
        win /= len(evs)
        alg = sum(alg_by.values())
        tname = tile_kernel_name(bt.info)
        kname = tname + "+splitkv_decode_kernel"
        ts = [traffic_per_launch(k, w.name) for k in tname.split("+")]
        t2 = traffic_per_launch(KERNEL_NAMES["splitkv_mma"], w.name)
        traffic = (sum(ts) + t2 if None not in ts and t2 is not None
                   else None)
        dom_ms = win
    else:
        dom = next(iter(alg_by))
        alg = alg_by[dom]
        kname = KERNEL_NAMES[dom]
        traffic = traffic_per_launch(kname, w.name)
        dom_ms = per_kernel[dom]
    achieved = alg / (dom_ms / 1e3) / 1e9
    return {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": alg,
            "ms_per_launch": round(dom_ms, 5)}


def per_config_line(w, dev, steps, warmup, peak, peak_kind, flush, cpu):
    """One of the other configurations, timed like the headline step (with
    an L2 flush before every step), with the oracle's rate beside it."""
    import torch
    from paged_kv_cache_attn_gb300 import harness as H
    cache = H.Cache(w, device=dev)
    bt = cache.batch().upload()
    q = torch.from_numpy(w.queries(bt.nb).view(np.int16)).to(dev) \
        .view(torch.bfloat16)
    out = torch.empty_like(q)
    uniq = unique_kv_bytes(bt.tables, bt.seq_lens, w.Hkv, w.d)
    ms, per_kernel, evs = time_steps(bt, q, out, steps, warmup, flush)
    roof = kernel_roofline(bt, w, per_kernel, evs, peak, peak_kind)
    gbs = uniq / (ms / 1e3) / 1e9
    res = {
        "description": w.description,
        "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d, "branches": bt.nb,
        "segments": int(len(bt.groups)), "unique_kv_bytes": uniq,
        "steps": steps, "ms_per_step": round(ms, 5),
        "value": round(gbs, 1), "unit": "GB/s",
        "branch_queries_per_s": round(bt.nb / (ms / 1e3), 1),
        "kernels_ms": {k: round(v, 5) for k, v in per_kernel.items()},
        "step_roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                          "peak": peak, "unit": "GB/s",
                          "frac": round(gbs / peak, 4)},
        "roofline": roof,
        "l2": "L2 flushed before every step (a 256 MB buffer written, then "
              "another 256 MB buffer read, so no dirty line is left); each "
              "step timed by its own events",
        "gpu_launches": kernels_per_step(bt.info) * steps,
    }
    if len(bt.groups):
        res["sharing_measured_ncu"] = measured_sharing(w.name)
    cache.close()
    if cpu:
        res["cpu_baseline"] = cpu_baseline(w, budget_s=5.0)
    return res


def run_ours(args):
    import torch
    from paged_kv_cache_attn_gb300 import binding as B
    from paged_kv_cache_attn_gb300 import harness as H
    from paged_kv_cache_attn_gb300 import workloads as W

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = f"cuda:{local if ws > 1 else 0}"
    torch.cuda.set_device(dev)
    w = W.make(args.workload, rank)
    cache = H.Cache(w, device=dev)
    bt = cache.batch().upload()
    nb = bt.nb
    q_host = w.queries(nb)
    q = torch.from_numpy(q_host.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty_like(q)
    uniq = unique_kv_bytes(bt.tables, bt.seq_lens, w.Hkv, w.d)
    stream = torch.cuda.current_stream()

    # Timed region: K steps (inputs far larger than L2, no flush), the
    # library's per-kernel events recorded on the launching streams.
    K = args.steps
    peak, peak_kind = measured_peaks()
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier = torch.distributed.barrier if ws > 1 else None
        ms_step, per_kernel, evs = time_steps(bt, q, out, K, args.warmup,
                                              before=barrier, after=barrier)
    if ws > 1:
        t = torch.tensor([ms_step], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_step = float(t.item())
    launches_per_step = kernels_per_step(bt.info)
    roof = kernel_roofline(bt, w, per_kernel, evs, peak, peak_kind)

    # End to end through the public API with host buffers.  Per step the
    # host builds the batch and the plan into pinned staging buffers
    # (allocated once, as an engine would), copies q / tables / lengths /
    # segments / plan host -> device, runs the step and copies the output
    # back.  Serial: each step waits for the previous one.  Pipelined (the
    # reported value): two sets of staging and device buffers; the host plans
    # step i + 1 and its inputs cross on a copy stream while the device runs
    # step i, and each step's output is read back once it is done -- what an
    # engine does when the next step's lengths and tables are known ahead
    # (kv_reserve).  Every step still moves all its inputs and its output.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mb = bt.tables.shape[1]

    def staging():
        p_ = {
            "q": torch.from_numpy(q_host.view(np.int16)).pin_memory(),
            "tables": torch.empty((nb, mb), dtype=torch.int32).pin_memory(),
            "lens": torch.empty(nb, dtype=torch.int32).pin_memory(),
            "groups": torch.empty((nb + 1) * 4, dtype=torch.int32).pin_memory(),
            "plan": torch.empty(2 * len(bt.plan) + 1024,
                                dtype=torch.int32).pin_memory(),
            "out": torch.empty((nb, w.Hq, w.d), dtype=torch.int16).pin_memory(),
        }
        d_ = {k: torch.empty_like(v, device=dev) for k, v in p_.items()}
        return p_, d_

    bufs = [staging(), staging()]
    wsb = [torch.empty(2 * bt.info.workspace_bytes + 4096, dtype=torch.uint8,
                       device=dev) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)   # host -> device
    back_stream = torch.cuda.Stream(device=dev)   # device -> host: its own
    # stream, so that the next step's inputs do not queue behind this
    # step's read-back (which waits for the step)
    h2d = d2h = 0

    def host_plan(pin):
        tables, lens, groups = B.kv_build_batch(
            cache.h, bt.ids, mb, pin["tables"].numpy(), pin["lens"].numpy(),
            pin["groups"].numpy())
        plan, info = B.paged_decode_plan(nb, w.Hq, w.Hkv, w.d, mb, lens,
                                         groups, sms,
                                         plan_out=pin["plan"].numpy())
        n_g = 4 * max(len(groups), 1)
        parts = [("q", pin["q"].numel()), ("tables", nb * mb), ("lens", nb),
                 ("groups", n_g), ("plan", len(plan))]
        return parts, info, len(groups)

    def h2d_copy(pin, dbf, parts):
        for k, n in parts:
            if dbf[k].dim() == 1:
                dbf[k][:n].copy_(pin[k][:n], non_blocking=True)
            else:
                dbf[k].copy_(pin[k], non_blocking=True)

    def decode_from(dbf, info, ng, ws_):
        B.paged_decode_attn(dbf["q"].view(torch.bfloat16), cache.k[0],
                            cache.v[0], w.num_blocks, dbf["tables"],
                            dbf["lens"], dbf["groups"], ng, nb, mb, w.Hq,
                            w.Hkv, w.d, w.scale,
                            dbf["out"].view(torch.bfloat16), dbf["plan"], info,
                            ws_, ws_.numel())

    # Serial.
    e2e_t = []
    for i in range(max(args.e2e_steps, 1) + 3):
        pin, dbf = bufs[0]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        parts, info, ng = host_plan(pin)
        h2d_copy(pin, dbf, parts)
        decode_from(dbf, info, ng, wsb[0])
        pin["out"].copy_(dbf["out"], non_blocking=True)
        torch.cuda.synchronize()
        if i >= 3:
            e2e_t.append(time.perf_counter() - t0)
        h2d = sum(n * 4 for _, n in parts[1:]) + pin["q"].numel() * 2
        d2h = pin["out"].numel() * 2
    e2e_serial_s = statistics.median(e2e_t)

    # Pipelined.
    comp = torch.cuda.current_stream()
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    dec_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    n_pipe = max(args.e2e_steps, 4)
    started = [False, False]
    t_start = None
    for i in range(n_pipe + 3):
        if i == 3:
            torch.cuda.synchronize()
            t_start = time.perf_counter()
        sl = i & 1
        pin, dbf = bufs[sl]
        if started[sl]:
            # The staging set is reused: its last H2D copy must have run,
            # and its last output must have been read back.
            h2d_done[sl].synchronize()
            d2h_done[sl].synchronize()
        parts, info, ng = host_plan(pin)
        with torch.cuda.stream(copy_stream):
            if started[sl]:
                copy_stream.wait_event(dec_done[sl])
            h2d_copy(pin, dbf, parts)
            h2d_done[sl].record(copy_stream)
        comp.wait_event(h2d_done[sl])
        decode_from(dbf, info, ng, wsb[sl])
        dec_done[sl].record(comp)
        with torch.cuda.stream(back_stream):
            back_stream.wait_event(dec_done[sl])
            pin["out"].copy_(dbf["out"], non_blocking=True)
            d2h_done[sl].record(back_stream)
        started[sl] = True
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t_start) / n_pipe

    # The same step with every branch re-reading its whole table (no
    # shared-prefix segments): time and bytes requested, for the sharing
    # criterion (prefix bytes moved shared vs per-branch re-read).
    sharing = None
    if len(bt.groups):
        bu = cache.batch(flags=B.KV_PLAN_IGNORE_GROUPS).upload()
        for _ in range(3):
            bu.decode(q, out)
        n_u = 20
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n_u):
            bu.decode(q, out)
        e1.record(stream)
        torch.cuda.synchronize()
        ms_u = e0.elapsed_time(e1) / n_u
        bytes_shared = sum(item_bytes(bt.plan, bt.info, w.Hkv, w.d,
                                      bt.seq_lens, k) for k in ("row", "tile"))
        bytes_unshared = item_bytes(bu.plan, bu.info, w.Hkv, w.d, bu.seq_lens,
                                    "row")
        # Prefix bytes: each branch re-reading every segment it is in,
        # against what the shared plan's segment items read.
        kvb = 2 * w.d * 2 * w.Hkv * 16  # bytes per block, all kv-heads
        pref_unshared = int(sum(int(g[1]) * int(g[3]) for g in bt.groups)) * kvb
        pref_shared = sum(item_bytes(bt.plan, bt.info, w.Hkv, w.d, bt.seq_lens,
                                     k, segments_only=True)
                          for k in ("row", "tile"))
        sharing = {
            "ms_per_step_shared": round(ms_step, 5),
            "ms_per_step_per_branch_reread": round(ms_u, 5),
            "speedup": round(ms_u / ms_step, 3),
            "bytes_requested_shared": bytes_shared,
            "bytes_requested_per_branch_reread": bytes_unshared,
            "prefix_bytes_shared": pref_shared,
            "prefix_bytes_per_branch_reread": pref_unshared,
            "prefix_bytes_factor": round(pref_unshared / max(pref_shared, 1), 2),
            "measured_ncu": measured_sharing(w.name),
        }

    # NEXT-1: each branch's newest token appended and attended to in one
    # launch vs a batched one-token append followed by the plain step.  Every
    # step adds one token per branch (a real decode loop); device time only.
    fused = None
    if args.fused_steps > 0:
        rng = np.random.default_rng(17)
        kst = torch.from_numpy(W.f32_to_bf16_bits(rng.standard_normal(
            (nb, w.Hkv, w.d), dtype=np.float32)).view(np.int16)).to(dev) \
            .view(torch.bfloat16)
        vst = kst.flip(0).contiguous()
        ids = cache.decode_ids
        ones = [1] * nb

        def ev():
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            return e

        # Each step needs up to one new block per branch every 16 tokens;
        # keep to what the pool's free blocks allow.
        free = len(B.kv_get_free_stack(cache.h))
        n_fused = max(1, min(args.fused_steps, 16 * free // (2 * nb) - 4))
        t_fused, t_unfused = [], []
        for i in range(n_fused + 2):
            B.kv_reserve(cache.h, ids, ones)
            bf = cache.batch().upload()
            e0 = ev()
            bf.decode_append(q, kst, vst, out)
            e1 = ev()
            torch.cuda.synchronize()
            if i >= 2:
                t_fused.append(e0.elapsed_time(e1))
        for i in range(n_fused + 2):
            e0 = ev()
            B.kv_append_batch(cache.h, ids, ones, kst, vst)
            e1 = ev()
            bu = cache.batch().upload()
            e2 = ev()
            bu.decode(q, out)
            e3 = ev()
            torch.cuda.synchronize()
            if i >= 2:
                t_unfused.append(e0.elapsed_time(e1) + e2.elapsed_time(e3))
        fused = {
            "steps": n_fused,
            "ms_fused_append_decode": round(statistics.median(t_fused), 5),
            "ms_append_then_decode": round(statistics.median(t_unfused), 5),
            "note": "device time per step (events around the launches); the "
                    "batch is rebuilt on the host between steps",
        }

    # NEXT-4: spill whole branches to pinned host memory and bring them back
    # (device <-> host over the CPU-GPU link), bandwidth of each direction.
    offload = None
    if args.offload_branches > 0:
        victims = [i for i in cache.decode_ids
                   if B.kv_branch_info(cache.h, i)["parent"] < 0]
        victims = victims[:args.offload_branches]
        nblk = sum(B.kv_branch_info(cache.h, i)["n_blocks"] for i in victims)
        if victims and nblk > 0:
            hshape = (w.num_layers, nblk, w.Hkv, w.block_size, w.d)
            hk = torch.empty(hshape, dtype=torch.bfloat16).pin_memory()
            hv = torch.empty(hshape, dtype=torch.bfloat16).pin_memory()
            B.kv_offload_attach(cache.h, hk, hv, nblk)
            byts = nblk * w.num_layers * w.Hkv * w.block_size * w.d * 2 * 2
            t_sp, t_re = [], []
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e2 = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                B.kv_spill(cache.h, victims)
                e1.record(stream)
                B.kv_restore(cache.h, victims)
                e2.record(stream)
                torch.cuda.synchronize()
                t_sp.append(e0.elapsed_time(e1))
                t_re.append(e1.elapsed_time(e2))
            # The link's own ceiling: one contiguous copy-engine copy of the
            # same pinned buffer each way (scattered blocks cannot beat it).
            dk = torch.empty_like(hk, device=dev)
            t_h2d, t_d2h = [], []
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e2 = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                dk.copy_(hk, non_blocking=True)
                e1.record(stream)
                hk.copy_(dk, non_blocking=True)
                e2.record(stream)
                torch.cuda.synchronize()
                t_h2d.append(e0.elapsed_time(e1))
                t_d2h.append(e1.elapsed_time(e2))
            del dk
            half = hk.numel() * hk.element_size()
            spill = byts / (min(t_sp) / 1e3) / 1e9
            restore = byts / (min(t_re) / 1e3) / 1e9
            link_d2h = half / (min(t_d2h) / 1e3) / 1e9
            link_h2d = half / (min(t_h2d) / 1e3) / 1e9
            offload = {
                "branches": len(victims), "blocks": nblk, "bytes": byts,
                "spill_gbs": round(spill, 1),
                "restore_gbs": round(restore, 1),
                "link_d2h_gbs": round(link_d2h, 1),
                "link_h2d_gbs": round(link_h2d, 1),
                "spill_frac_of_link": round(spill / link_d2h, 3),
                "restore_frac_of_link": round(restore / link_h2d, 3),
                "note": "one copy kernel per direction, device pool <-> "
                        "pinned host memory; best of 3.  link_*: a "
                        "contiguous copy-engine copy of the pinned K buffer "
                        "each way, the CPU-GPU link's ceiling",
            }
        # Prefetch: the spilled branches come back on a side stream while the
        # step keeps decoding the branches that stayed resident (their batch
        # is built before the restore and references none of the device
        # blocks it pops).  As many steps as one restore takes.
        gone = set(victims)
        others = ([i for i in cache.decode_ids if i not in gone]
                  if victims and nblk > 0 else [])
        if others:
            B.kv_spill(cache.h, victims)
            torch.cuda.synchronize()
            bo = cache.batch(ids=others).upload()
            qo = q[:len(others)]
            oo = torch.empty_like(qo)
            n_dec = max(1, int(round(min(t_re) / ms_step)))

            def decode_steps():
                d0 = torch.cuda.Event(enable_timing=True)
                d1 = torch.cuda.Event(enable_timing=True)
                d0.record(stream)
                for _ in range(n_dec):
                    bo.decode(qo, oo)
                d1.record(stream)
                return d0, d1

            bo.decode(qo, oo)
            torch.cuda.synchronize()
            a0, a1 = decode_steps()
            torch.cuda.synchronize()
            side = torch.cuda.Stream(device=dev)
            r0 = torch.cuda.Event(enable_timing=True)
            r1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(side):
                r0.record(side)
                B.kv_restore(cache.h, victims, stream=side)
                r1.record(side)
            b0, b1 = decode_steps()
            torch.cuda.synchronize()
            t_r = r0.elapsed_time(r1)
            offload["prefetch"] = {
                "resident_branches": len(others), "decode_steps": n_dec,
                "ms_per_step_alone": round(a0.elapsed_time(a1) / n_dec, 5),
                "ms_per_step_beside_restore":
                    round(b0.elapsed_time(b1) / n_dec, 5),
                "restore_ms_beside_decode": round(t_r, 4),
                "restore_gbs_beside_decode": round(byts / (t_r / 1e3) / 1e9, 1),
                "note": "the spilled branches restored on a side stream while "
                        "the resident branches decode on the main stream",
            }

    # The same step captured once into a CUDA graph and replayed: what an
    # engine launching many layers per token would do; it removes the host's
    # per-launch cost, which matters when the step itself is short.
    graph = None
    try:
        qg = q.clone()
        og = torch.empty_like(out)
        bt.decode(qg, og)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            bt.decode(qg, og)
        for _ in range(3):
            cg.replay()
        n_g = max(20, min(K, 500))
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        g0.record(stream)
        for _ in range(n_g):
            cg.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        ms_g = g0.elapsed_time(g1) / n_g
        graph = {"ms_per_step": round(ms_g, 5),
                 "value": round(uniq / (ms_g / 1e3) / 1e9, 1),
                 "unit": "GB/s", "replays": n_g}
    except RuntimeError as exc:          # capture unsupported: report why
        graph = {"unavailable": str(exc)[:200]}

    # NEXT-3: the same step over an e4m3 copy of the workload's pool (codes
    # plus one 16-byte scale record per block and kv-head).
    e4m3 = None
    if args.e4m3_steps > 0:
        c8 = H.Cache(w, device=dev, kv_dtype="e4m3")
        b8 = c8.batch().upload()
        uniq8 = unique_kv_bytes(b8.tables, b8.seq_lens, w.Hkv, w.d, elem=1,
                                record=16)
        for _ in range(3):
            b8.decode(q, out)
        torch.cuda.synchronize()
        K8 = args.e4m3_steps
        ev8 = [[torch.cuda.Event(enable_timing=True) for _ in range(6)]
               for _ in range(K8)]
        for row in ev8:
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
        s8 = torch.cuda.Event(enable_timing=True)
        t8 = torch.cuda.Event(enable_timing=True)
        s8.record(stream)
        for i in range(K8):
            B.kv_set_launch_events(ev8[i])
            b8.decode(q, out)
        t8.record(stream)
        B.kv_set_launch_events(None)
        torch.cuda.synchronize()
        code8, det8 = b8.device_status()
        if code8:
            raise RuntimeError(f"e4m3 device status {code8} ({det8})")
        ms8 = s8.elapsed_time(t8) / K8
        has_t = b8.info.n_tile_items > 0
        has_r = b8.info.n_row_items > 0
        k8ms = {}
        if has_t:
            k8ms["tile_e4m3"] = sum(e[0].elapsed_time(e[1]) for e in ev8) / K8
        if has_r:
            k8ms["splitkv_e4m3"] = sum(e[2].elapsed_time(e[3]) for e in ev8) / K8
        k8ms["lse_merge"] = sum(e[4].elapsed_time(e[5]) for e in ev8) / K8
        alg8 = sum(item_bytes(b8.plan, b8.info, w.Hkv, w.d, b8.seq_lens, k,
                              elem=1, record=16)
                   for k, on in (("row", has_r), ("tile", has_t)) if on)
        if has_t and has_r:        # the two passes' common window
            win8 = sum(max(e[0].elapsed_time(e[1]), e[0].elapsed_time(e[3])) -
                       min(0.0, e[0].elapsed_time(e[2])) for e in ev8) / K8
            kname8 = "tile_e4m3_kernel+splitkv_e4m3_kernel"
        else:
            win8 = k8ms["tile_e4m3" if has_t else "splitkv_e4m3"]
            kname8 = "tile_e4m3_kernel" if has_t else "splitkv_e4m3_kernel"
        ach8 = alg8 / (win8 / 1e3) / 1e9
        tr8 = [traffic_per_launch(n, w.name) for n, on in
               (("tile_e4m3_kernel", has_t), ("splitkv_e4m3_kernel", has_r)) if on]
        traffic8 = sum(tr8) if tr8 and None not in tr8 else None
        e4m3 = {
            "ms_per_step": round(ms8, 5),
            "unique_kv_bytes": uniq8,
            "value": round(uniq8 / (ms8 / 1e3) / 1e9, 1),
            "unit": "GB/s (unique e4m3 KV bytes / step time)",
            "branch_queries_per_s": round(nb / (ms8 / 1e3), 1),
            "speedup_vs_bf16_step": round(ms_step / ms8, 3),
            "kernels_ms": {k: round(v, 5) for k, v in k8ms.items()},
            "roofline": {
                "kernel": kname8, "bound": "hbm",
                "achieved": round(ach8, 1), "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(ach8 / peak, 4),
                "traffic": traffic8,
                "algorithmic_bytes_per_launch": alg8,
                "ms_per_launch": round(win8, 5),
                "note": "e4m3 codes + 16-byte scale record per block read; "
                        "with both passes, their common window"},
            "steps": K8,
        }
        c8.close()

    # The other configurations, each timed on its own (N = 1 only), with the
    # oracle's rate on the host cores beside each, and the oracle's
    # single-thread rate on the Llama-3-8B-shaped one.
    per_config = None
    if args.per_config_steps > 0 and ws == 1:
        flush = [torch.zeros(64 << 20, dtype=torch.float32, device=dev)
                 for _ in range(2)]
        per_config = {}
        for name in ("tiny_tree", "independent", "fanout", "deep_tree"):
            per_config[name] = per_config_line(
                W.make(name, rank), dev, args.per_config_steps, args.warmup,
                peak, peak_kind, flush, not args.no_cpu_baseline)
        if not args.no_cpu_baseline:
            st = cpu_baseline(W.make("independent", rank), budget_s=6.0,
                              threads=1)
            per_config["independent"]["cpu_baseline_single_thread"] = st
        del flush

    res = None
    if rank == 0:
        clocks = clk.summary()
        res = {
            "metric": METRIC,
            "value": round(uniq * ws / (ms_step / 1e3) / 1e9, 1),
            "unit": "GB/s",
            "n_gpus": ws,
            "steps": K,
            "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "branch_queries_per_s": round(nb * ws / (ms_step / 1e3), 1),
            "config": {
                "workload": w.name,
                "description": w.description,
                "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d, "block_size": 16,
                "branches": nb,
                "unique_kv_bytes": uniq,
                "segments": int(len(bt.groups)),
                "l2": "inputs larger than L2 (unique KV far above 129 MB); "
                      "no flush",
                "parallelism": f"replicas x{ws}",
            },
            "kernels_ms": {k: round(v, 5) for k, v in per_kernel.items()},
            "roofline": roof,
            "step_roofline": {
                "bound": "hbm",
                "achieved": round(uniq / (ms_step / 1e3) / 1e9, 1),
                "peak": peak,
                "unit": "GB/s",
                "frac": round(uniq / (ms_step / 1e3) / 1e9 / peak, 4),
                "note": "unique KV bytes of the whole step / step time",
            },
            "e2e": {
                "value": round(uniq / e2e_s / 1e9, 1),
                "unit": "GB/s",
                "ms_per_step": round(e2e_s * 1e3, 4),
                "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "mode": "pipelined: host plan and H2D of step i+1 overlap "
                        "step i on the device; each step's output read back "
                        "on a stream of its own",
                "serial_value": round(uniq / e2e_serial_s / 1e9, 1),
                "serial_ms_per_step": round(e2e_serial_s * 1e3, 4),
            },
            "sharing": sharing,
            "fused_append": fused,
            "radix_index": radix_timing(),
            "offload": offload,
            "graph_replay": graph,
            "kv_e4m3": e4m3,
            "per_config": per_config,
            "gpu_launches": launches_per_step * K,
            "clocks": clocks,
        }
        if not args.no_cpu_baseline and ws == 1:
            res["cpu_baseline"] = cpu_baseline(w)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    cache.close()
    return res


def run_reference(args):
    """The fp64 oracle on host threads; each step one bounded sample."""
    from paged_kv_cache_attn_gb300 import workloads as W
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    w = W.CONFIGS[args.workload]()
    sample, nb = prepare_sample(w, 16)
    units = [(i, g) for i in range(len(sample)) for g in range(w.Hkv)]
    np.random.default_rng(3).shuffle(units)
    cores = min(host_cores(), len(units))
    # Size a step so the whole run takes about two minutes.
    t0 = time.perf_counter()
    oracle_unit(w, sample[units[0][0]], units[0][1])
    unit_s = max(time.perf_counter() - t0, 1e-4)
    per_step = 120.0 / (args.steps + args.warmup)
    per = max(1, min(len(units), int(per_step * cores / unit_s)))
    times, byts, pos = [], [], 0
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        for i in range(args.warmup + args.steps):
            chunk = [units[(pos + j) % len(units)] for j in range(per)]
            pos += per
            t0 = time.perf_counter()
            b = run_units(w, sample, chunk, min(cores, per), ex)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
                byts.append(b)
    total_t = sum(times)
    val = sum(byts) / total_t / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 4),
        "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_t / len(times) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description},
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s",
                         "cores": min(cores, per), "kind": "oracle",
                         "sample": f"{per} (branch, kv-head) units per step "
                                   f"from {len(sample)} of {nb} branches of "
                                   f"{w.name}, fp64 numpy",
                         "cpu": cpu_model()},
        "e2e": {"value": round(val, 4), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def radix_timing():
    """Host cost of the radix prefix index on a multi-turn workload: 256
    conversations sharing a 2048-token system prompt, each inserted after its
    turn and matched at the next turn (µs per call)."""
    from paged_kv_cache_attn_gb300 import binding as B
    h = B.kv_pool_create(200000, 1, 1, 128)
    r = B.kv_radix_create(h)
    rng = np.random.default_rng(21)
    prompt = rng.integers(0, 32000, 2048).tolist()
    convs = [prompt + rng.integers(0, 32000, 256).tolist() for _ in range(256)]
    t_ins = t_match = 0.0
    for turn in range(2):
        for i, c in enumerate(convs):
            t0 = time.perf_counter()
            B.kv_radix_match(r, c)
            t_match += time.perf_counter() - t0
            b = B.kv_branch_create(h)
            B.kv_append(h, b, len(c))
            t0 = time.perf_counter()
            B.kv_radix_insert(r, b, c)
            t_ins += time.perf_counter() - t0
            B.kv_free(h, b)
            convs[i] = c + rng.integers(0, 32000, 128).tolist()
    n = 2 * len(convs)
    nodes = B.kv_radix_num_nodes(r)
    B.kv_radix_destroy(r)
    B.kv_pool_destroy(h)
    return {"match_us": round(t_match / n * 1e6, 1),
            "insert_us": round(t_ins / n * 1e6, 1), "nodes": nodes,
            "workload": "256 conversations, 2048-token shared prompt, 2 turns "
                        "(2304 then 2432 tokens), through the Python binding"}


def profile_step(args):
    """A few decode steps of one workload and one plan, nothing else."""
    import torch
    from paged_kv_cache_attn_gb300 import binding as B
    from paged_kv_cache_attn_gb300 import harness as H
    from paged_kv_cache_attn_gb300 import workloads as W
    w = W.make(args.workload)
    cache = H.Cache(w, device="cuda:0")
    flags = B.KV_PLAN_IGNORE_GROUPS if args.profile_step == "reread" else 0
    bt = cache.batch(flags=flags).upload()
    q = torch.from_numpy(w.queries(bt.nb).view(np.int16)).cuda() \
        .view(torch.bfloat16)
    out = torch.empty_like(q)
    for _ in range(args.steps):
        bt.decode(q, out)
    torch.cuda.synchronize()
    code, detail = bt.device_status()
    if code:
        raise RuntimeError(f"device status {code} ({detail})")
    print(json.dumps({"workload": w.name, "plan": args.profile_step,
                      "tile_items": bt.info.n_tile_items,
                      "split_items": bt.info.n_row_items,
                      "steps": args.steps}))
    cache.close()


def main():
    args = parse()
    if args.profile_step:
        profile_step(args)
        return
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res, default=lambda o: o.item() if hasattr(o, "item")
                         else str(o)), flush=True)


if __name__ == "__main__":
    main()
