"""Benchmark: paged decode attention on the Llama-3.1-8B-shaped GQA layer.

One step = pa_reshape_and_cache of the batch's 256 new tokens + pa_decode of
256 sequences (32 q heads / 8 kv heads, head_dim 128, bf16, block size 16,
contexts U[512, 4096], blocks scattered over a 100,000-block pool). Two such
batches over disjoint blocks of the same pool alternate step by step, and each
step reads ~2.4 GB of K/V, far more than the 129 MB L2, so no step starts with
its inputs in L2.

Prints one JSON line. ``value`` is the algorithmic HBM throughput of the step
(K/V bytes of every attended token + q + out + the new rows written) over the
device time; ``e2e`` is the same metric through the public Python API with the
step's host inputs copied in from pinned memory and the output copied back
inside the timed region (overlapped with the neighbouring steps as a serving
loop would, and ``e2e.serial`` with nothing overlapped). At one GPU the line
also carries ``workloads``: each other configuration (tiny, OPT-13B MHA, the
Llama batch over E4M3 codes, 70B-shaped GQA-8 on short contexts, the
shared-prefix batches with plain and cascade decode, the 32K-128K contexts at
block 16 and 32, the copy-on-write copies) device-timed on its own, with its
attention call's roofline, clocks and a bounded oracle sample. ``--headline-only``
skips them.

``--impl reference`` times the CPU oracle (the only reference this method has)
on bounded samples of the same workload.

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path has no exchange step), the timed region is bracketed by barriers and the
slowest rank's time is used; ``value`` aggregates all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and seqs/s, 1 GPU"
WORKLOAD = ("Llama-3.1-8B GQA decode layer: 256 seqs x (32 q / 8 kv heads, d 128), bf16, block 16, "
            "context U[512,4096], 100k-block shuffled pool; step = reshape_and_cache(256 new tokens) + decode")
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle sample")
    ap.add_argument("--profile", action="store_true",
                    help="run only the step's kernels on a 64-sequence batch of the same shape (for ncu)")
    ap.add_argument("--profile-fp8", action="store_true",
                    help="the same 64-sequence case with an E4M3 cache (for ncu)")
    ap.add_argument("--profile-case", choices=["split", "cascade", "cascade_x16", "mha", "g8", "copy", "reshape"],
                    default=None,
                    help="a small case of another path for ncu: split (2 seqs, 48K-64K tokens, 64 q / 8 kv), "
                         "cascade (32 prompts x 8 samples), mha (the OPT-13B batch), g8 (64 seqs of the "
                         "64 q / 8 kv short-context batch, plain decode)")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other configurations' entries ('workloads') of the default run")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="write profiles/pa_decode_llama8b.json from `ncu --page raw --csv` of the --profile case")
    ap.add_argument("--workload", default="llama8b",
                    choices=["llama8b", "tiny", "opt13b", "shared", "shared_cow", "long70b_b16", "long70b_b32",
                             "llama8b_fp8", "long70b_b16_fp8", "shared_cascade", "shared_cow_cascade", "gemma_d256",
                             "llama70b_short", "llama70b_short_fp8",
                             "shared_x16", "shared_x16_cascade", "shared_x32", "shared_x32_cascade",
                             "llama8b_nhd", "llama8b_fp8_nhd", "long70b_b16_nhd", "shared_cascade_nhd",
                             "llama8b_s2048", "llama8b_s2048_fp8",
                             "copy_blocks", "swap_out", "swap_in", "reshape", "reshape_prefill"],
                    help="the other workload shapes give a device-timed line of their own (no e2e / CPU legs); "
                         "a _nhd suffix stores the pools NHD")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------
def dist_init(n):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------
def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources that define and launch the timed decode kernel (16-bit cache): the
# ncu counters in the profile summary stay valid while none of these changes.
DECODE_KERNEL_SOURCES = ("pa_api.cu", "pa_decode.cuh", "pa_decode_bf16.cu", "pa_decode_launch.cuh",
                         "pa_device.cuh", "pa_internal.h")


def kernel_source_sha():
    """Hash of the decode kernel's sources with comments and whitespace removed
    (a comment edit does not change the kernel the counters were taken on)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_04_gb300", "csrc")
    for name in DECODE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode() + " ".join(text.split()).encode())
    return h.hexdigest()


PROFILE_RECORD = os.path.join(ROOT, "profiles", "pa_decode_llama8b.json")


def profiled_traffic():
    """DRAM bytes per pa_decode launch of the benchmark batch, from the record that
    ``--record-traffic`` wrote from an ncu capture, while it matches the kernel sources."""
    try:
        with open(PROFILE_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_sha():
        return None
    return {"bytes": float(rec["traffic_bytes_per_launch"]),
            "source": f"ncu capture of the {rec['capture_case']} ({rec['scale']:.4f} x its per-launch traffic "
                      f"scaled by algorithmic bytes), profiles/pa_decode_llama8b.json"}


def record_traffic(csv_path):
    """Write profiles/pa_decode_llama8b.json from ``ncu --page raw --csv`` of the profiling
    case (``--profile``): its dram read + write bytes per launch, scaled to the benchmark
    batch's launch by algorithmic bytes (traffic grows with the tokens read)."""
    import csv
    from paged_kv_cache_04_gb300 import roofline, workloads
    rows = list(csv.reader(open(csv_path)))
    head = rows[0]
    data = [r for r in rows[2:] if r and "paged_decode_kernel" in ",".join(r)]
    if not data:
        raise SystemExit(f"no paged_decode_kernel row in {csv_path}")
    r = data[-1]
    col = {n: i for i, n in enumerate(head)}
    unit_scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    units = rows[1]

    def val(name):
        i = col[name]
        return float(r[i].replace(",", "")) * unit_scale.get(units[i], 1)
    small = workloads.llama8b(device="cpu", S=64, num_blocks=16_000)
    full = workloads.llama8b(device="cpu")
    small_bytes = roofline.decode_bytes(small.context_lens.tolist(), 32, 8, 128, 2)
    full_bytes = roofline.decode_bytes(full.context_lens.tolist(), 32, 8, 128, 2)
    traffic = val("dram__bytes_read.sum") + val("dram__bytes_write.sum")
    rec = {"kernel": "paged_decode_kernel<bf16, bf16, bf16, 128, tensor-core path, plain mode>",
           "capture_case": "64-sequence profiling case (bench.py --profile)",
           "dram_bytes_per_launch_small": traffic, "algorithmic_bytes_small": small_bytes,
           "scale": traffic / small_bytes, "algorithmic_bytes_full": full_bytes,
           "traffic_bytes_per_launch": round(traffic / small_bytes * full_bytes),
           "gpu_time_ns_small": val("gpu__time_duration.sum"), "source_sha256": kernel_source_sha(),
           "csv": os.path.basename(csv_path)}
    with open(PROFILE_RECORD, "w") as f:
        json.dump(rec, f, indent=1)
    print(json.dumps(rec))


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------
def make_batches(device):
    import torch
    from paged_kv_cache_04_gb300 import workloads
    a = workloads.llama8b(device=device)
    b = workloads.llama8b(device=device, rotate=50_000)
    b.k_cache, b.v_cache = a.k_cache, a.v_cache   # one pool, two disjoint block sets
    used_a = set(a.block_tables[a.block_tables >= 0].tolist())
    used_b = set(b.block_tables[b.block_tables >= 0].tolist())
    assert not used_a & used_b, "the two batches must not share blocks"
    torch.cuda.synchronize()
    return [a, b]


def step_bytes(wl):
    from paged_kv_cache_04_gb300 import roofline
    ctx = wl.context_lens.tolist()
    dec = roofline.decode_bytes(ctx, wl.H, wl.G, wl.d, 2)
    rc = roofline.reshape_and_cache_bytes(wl.slot_mapping.numel(), wl.G, wl.d, 2)
    return dec, rc, sum(ctx)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local):
    import torch
    import paged_kv_cache_04_gb300 as pa
    from paged_kv_cache_04_gb300 import _build
    if rank == 0 or not os.path.exists(pa.library_path):
        _build.ensure_built()
    barrier(world)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pa.library()
    batches = make_batches(dev)
    outs = [torch.empty_like(wl.q) for wl in batches]
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        wl = batches[i % 2]
        pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
        if ev is not None:
            ev[0].record(stream)
        pa.pa_decode(outs[i % 2], wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
        if ev is not None:
            ev[1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if pa.pa_get_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(t0.elapsed_time(t1), world, dev)
    # The decode kernel's own launch time, from a second pass of the same steps with
    # events around each decode call (kept out of the pass above: an event between the
    # cache write and the decode stops the decode from being scheduled early).
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        step(i, dec_ev[i])
    torch.cuda.synchronize()
    dec_ms = [a.elapsed_time(b) for a, b in dec_ev]

    # end to end through the public API: pinned host inputs in, output back out
    host = []
    for wl in batches:
        h = {k: getattr(wl, k).cpu().pin_memory() for k in
             ("q", "new_key", "new_value", "slot_mapping", "block_tables", "context_lens")}
        h["out"] = torch.empty(wl.q.shape, dtype=wl.q.dtype).pin_memory()
        d = {k: torch.empty_like(getattr(wl, k)) for k in h if k != "out"}
        host.append((h, d))
    h2d = sum(v.numel() * v.element_size() for k, v in host[0][0].items() if k != "out")
    d2h = host[0][0]["out"].numel() * host[0][0]["out"].element_size()

    # As a serving loop would: step i's inputs go up on an upload stream while step
    # i - 1 computes, and its output comes back on a download stream; events keep
    # each double-buffered input / output pair from being reused too early.
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    fetched = [torch.cuda.Event() for _ in range(2)]
    for j in range(2):  # every buffer starts free
        computed[j].record(stream)
        fetched[j].record(stream)

    def e2e_step(i):
        j = i % 2
        wl = batches[j]
        h, d = host[j]
        with torch.cuda.stream(up):
            up.wait_event(computed[j])  # step i - 2 has finished reading these device inputs
            for k in d:
                d[k].copy_(h[k], non_blocking=True)
            in_ready[j].record(up)
        stream.wait_event(in_ready[j])
        stream.wait_event(fetched[j])  # step i - 2's output has left this buffer
        pa.pa_reshape_and_cache(d["new_key"], d["new_value"], wl.k_cache, wl.v_cache, d["slot_mapping"])
        pa.pa_decode(outs[j], d["q"], wl.k_cache, wl.v_cache, d["block_tables"], d["context_lens"], wl.scale)
        computed[j].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[j])
            h["out"].copy_(outs[j], non_blocking=True)
            fetched[j].record(down)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    K2 = max(20, K // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    up.wait_event(e0)
    for i in range(K2):
        e2e_step(i)
    stream.wait_event(fetched[(K2 - 1) % 2])  # the last output is on the host
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    # The same end-to-end step with nothing overlapped: one stream, copy in -> cache
    # write -> decode -> copy out, each step after the last (the latency of one step).
    def serial_step(i):
        j = i % 2
        wl = batches[j]
        h, d = host[j]
        for k in d:
            d[k].copy_(h[k], non_blocking=True)
        pa.pa_reshape_and_cache(d["new_key"], d["new_value"], wl.k_cache, wl.v_cache, d["slot_mapping"])
        pa.pa_decode(outs[j], d["q"], wl.k_cache, wl.v_cache, d["block_tables"], d["context_lens"], wl.scale)
        h["out"].copy_(outs[j], non_blocking=True)

    for i in range(3):
        serial_step(i)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    s0.record(stream)
    for i in range(K2):
        serial_step(i)
    s1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    serial_ms = max_over_ranks(s0.elapsed_time(s1), world, dev)
    clk = clocks.stop()
    for j in range(2):  # the overlapped copies delivered each batch's output
        if not torch.equal(host[j][0]["out"], outs[j].cpu()):
            raise RuntimeError("end-to-end output on the host differs from the device output")
    err = pa.pa_get_error()
    if err:
        raise RuntimeError(f"device error word set: {err}")

    stats = [step_bytes(wl) for wl in batches]
    dec_bytes = sum(s[0] for s in stats) / 2
    rc_bytes = sum(s[1] for s in stats) / 2
    tokens = sum(s[2] for s in stats) / 2
    S = batches[0].S
    ms_step = ms_total / K
    value = world * (dec_bytes + rc_bytes) / (ms_step * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    dec_avg = statistics.mean(dec_ms)
    achieved = dec_bytes / (dec_avg * 1e-3) / 1e9
    traffic = profiled_traffic()
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) K/V/q; no dataset)",
        "config": {"workload": WORKLOAD, "seqs": S, "q_heads": 32, "kv_heads": 8, "head_dim": 128,
                   "block_size": 16, "pool_blocks": batches[0].num_blocks,
                   "l2": "inputs larger than L2: ~2.4 GB of K/V per step, two batches on disjoint blocks alternate",
                   "parallelism": f"replicas x{world} (no exchange on the path)"},
        "seqs_per_s": round(world * S / (ms_step * 1e-3), 1),
        "kv_tokens_per_s": round(world * tokens / (ms_step * 1e-3), 1),
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "frac_of_nominal_peak": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"kernel": "paged_decode_kernel (pa_decode)", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic": traffic["bytes"] if traffic else None,
                     "traffic_source": traffic["source"] if traffic else
                     "null: no ncu capture of the current kernel sources",
                     "algorithmic_bytes_per_launch": int(dec_bytes),
                     "avg_launch_ms": round(dec_avg, 5)},
        "e2e": {"value": round(world * (dec_bytes + rc_bytes) / (e2e_ms / K2 * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms / K2, 5), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "how": "pinned host inputs up on one stream while the previous step computes, output down on a third",
                "serial": {"value": round(world * (dec_bytes + rc_bytes) / (serial_ms / K2 * 1e-3) / 1e9, 1),
                           "ms_per_step": round(serial_ms / K2, 5),
                           "how": "one stream: copy in, cache write, decode, copy out, step after step"}},
        "gpu_launches": 2 * K,  # the timed pass: one cache write and one decode per step
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(batches[0], args.cpu_seconds)
        line["cpu_baseline"]["one_thread"] = cpu_baseline(batches[0], args.cpu_seconds / 4, threads=1)
    if rank == 0 and world == 1 and not args.headline_only:
        # the other configurations, each timed on its own after the headline (N = 1 only)
        del batches, outs, host
        torch.cuda.empty_cache()
        extras = {}
        for name in EXTRA_WORKLOADS:
            # one entry's failure is recorded in that entry; the headline and the others stand
            try:
                extras[name] = measure_workload(name, max(10, min(30, K)), max(3, args.warmup),
                                                None if args.no_cpu_baseline else 2.0, local)
            except Exception as e:  # noqa: BLE001
                extras[name] = {"workload": name, "error": f"{type(e).__name__}: {e}"[:300]}
            torch.cuda.empty_cache()
        line["workloads"] = extras
    return line


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(wl, seqs):
    """Host copies of the sample's blocks, tables remapped, new tokens kept; no kernel touched them."""
    import torch
    B = wl.B
    bt = wl.block_tables.cpu()
    ctx = wl.context_lens.cpu()
    blocks = sorted({int(b) for s in seqs for b in bt[s, :-(-int(ctx[s]) // B)].tolist()})
    remap = {b: i for i, b in enumerate(blocks)}
    idx = torch.tensor(blocks, dtype=torch.long, device=wl.k_cache.device)
    k = wl.k_cache.index_select(0, idx).cpu()
    v = wl.v_cache.index_select(0, idx).cpu()
    nbt = torch.full((len(seqs), bt.shape[1]), -1, dtype=torch.int32)
    for i, s in enumerate(seqs):
        n = -(-int(ctx[s]) // B)
        nbt[i, :n] = torch.tensor([remap[int(b)] for b in bt[s, :n].tolist()], dtype=torch.int32)
    slots = wl.slot_mapping.cpu()
    new_slots = torch.tensor([remap[int(slots[s]) // B] * B + int(slots[s]) % B for s in seqs],
                             dtype=torch.int64)
    return dict(q=wl.q.cpu()[seqs], k=k, v=v, bt=nbt, ctx=ctx[seqs].clone(),
                key=wl.new_key.cpu()[seqs], value=wl.new_value.cpu()[seqs], slots=new_slots, scale=wl.scale)


def oracle_step(smp, threads):
    """The oracle's version of one step on the sample: write the new tokens, then attend."""
    import numpy as np
    import torch
    import oracle
    kb, vb = oracle.reshape_and_cache(smp["key"], smp["value"], smp["k"], smp["v"], smp["slots"])
    k = torch.from_numpy(np.ascontiguousarray(kb).view(np.int16)).view(torch.bfloat16)
    v = torch.from_numpy(np.ascontiguousarray(vb).view(np.int16)).view(torch.bfloat16)
    return oracle.decode(smp["q"], k, v, smp["bt"], smp["ctx"], smp["scale"], num_threads=threads)


def sample_bytes(smp):
    from paged_kv_cache_04_gb300 import roofline
    ctx = smp["ctx"].tolist()
    return (roofline.decode_bytes(ctx, 32, 8, 128, 2) + roofline.reshape_and_cache_bytes(len(ctx), 8, 128, 2))


def cpu_baseline(wl, seconds, threads=None):
    import oracle
    threads = threads or len(os.sched_getaffinity(0))
    n = 2
    while True:
        smp = oracle_sample(wl, list(range(n)))
        t = time.perf_counter()
        oracle_step(smp, threads)
        dt = time.perf_counter() - t
        if dt >= seconds or n >= wl.S:
            break
        n = min(wl.S, max(n + 1, int(n * min(8.0, 1.2 * seconds / max(dt, 1e-3)))))
    return {"value": round(sample_bytes(smp) / dt / 1e9, 4), "unit": "GB/s", "cores": min(threads, oracle.max_threads()),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"first {n} of {wl.S} sequences of the same batch (all 32 heads, its new tokens written "
                      f"first), float64 C oracle, OpenMP over (sequence, head), {threads} thread(s)"}


def run_reference(args, rank, world, local):
    import torch
    if rank != 0:
        return None
    threads = len(os.sched_getaffinity(0))
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    from paged_kv_cache_04_gb300 import workloads
    wl = workloads.llama8b(device=dev)
    # calibrate the per-step sample so the whole run takes about a minute
    budget = 60.0 / max(1, args.steps + args.warmup)
    smp = oracle_sample(wl, [0])
    t = time.perf_counter()
    oracle_step(smp, threads)
    one = time.perf_counter() - t
    n = max(1, min(wl.S, int(budget / max(one, 1e-6))))
    smp = oracle_sample(wl, list(range(n)))
    for _ in range(args.warmup):
        oracle_step(smp, threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(smp, threads)
    dt = (time.perf_counter() - t) / max(1, args.steps)
    value = sample_bytes(smp) / dt / 1e9
    import oracle
    cores = min(threads, oracle.max_threads())
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) K/V/q; no dataset)",
        "config": {"workload": WORKLOAD, "seqs": 256, "q_heads": 32, "kv_heads": 8, "head_dim": 128,
                   "block_size": 16, "pool_blocks": wl.num_blocks,
                   "l2": "n/a (CPU oracle)", "parallelism": "rank 0 only"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of 256 sequences per step (all 32 heads, new tokens written first)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def decode_oracle_baseline(wl, seconds, fp8=False):
    """The oracle's decode (float64, all host cores) on the first sequences of a workload,
    grown until one call takes about ``seconds``: GB/s of the same algorithmic bytes."""
    import torch
    import oracle
    from oracle import fp8 as ofp8
    from paged_kv_cache_04_gb300 import roofline
    threads = len(os.sched_getaffinity(0))
    B = wl.B
    bt_all, ctx_all = wl.block_tables.cpu(), wl.context_lens.cpu()
    n = 1
    while True:
        seqs = list(range(n))
        blocks = sorted({int(b) for s in seqs for b in bt_all[s, :-(-int(ctx_all[s]) // B)].tolist()})
        remap = {b: i for i, b in enumerate(blocks)}
        idx = torch.tensor(blocks if blocks else [0], dtype=torch.long, device=wl.k_cache.device)
        k, v = wl.k_cache.index_select(0, idx).cpu(), wl.v_cache.index_select(0, idx).cpu()
        bt = torch.full((n, bt_all.shape[1]), -1, dtype=torch.int32)
        for i, s in enumerate(seqs):
            m = -(-int(ctx_all[s]) // B)
            bt[i, :m] = torch.tensor([remap[int(b)] for b in bt_all[s, :m].tolist()], dtype=torch.int32)
        q, ctx = wl.q.cpu()[seqs], ctx_all[seqs].clone()
        t = time.perf_counter()
        if fp8:
            ofp8.decode(q, k.numpy(), v.numpy(), bt, ctx, wl.scale, wl.meta["k_scale"], wl.meta["v_scale"],
                        num_threads=threads, layout=wl.layout)
        else:
            oracle.decode(q, k, v, bt, ctx, wl.scale, num_threads=threads, layout=wl.layout)
        dt = time.perf_counter() - t
        if dt >= seconds or n >= wl.S:
            break
        n = min(wl.S, max(n + 1, int(n * min(8.0, 1.2 * seconds / max(dt, 1e-3)))))
    ke = wl.k_cache.element_size()
    byt = (roofline.decode_bytes(ctx.tolist(), wl.H, wl.G, wl.d, ke) - 2 * n * wl.H * wl.d * ke
           + 2 * n * wl.H * wl.d * wl.q.element_size())
    return {"value": round(byt / dt / 1e9, 4), "unit": "GB/s", "cores": min(threads, oracle.max_threads()),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"decode of the first {n} of {wl.S} sequences, float64 oracle, OpenMP over (sequence, head)"}


def time_steps(step, steps, warmup, flush):
    """Mean CUDA-event time (ms) of ``step`` after warm-up, reading ``flush`` (larger than L2) between steps."""
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    torch.cuda._sleep(int(2e6 * (2 + steps)))
    times = []
    for _ in range(steps):
        flush.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(x.elapsed_time(y) for x, y in times)


def measure_cache_workload(name, steps, warmup, cpu_seconds=None, clocks_index=0):
    """The cache kernels on their own: CoW block copies, swap to and from pinned host
    memory, and the cache write at decode and at prefill size."""
    import numpy as np
    import torch
    import paged_kv_cache_04_gb300 as pa
    import oracle
    from paged_kv_cache_04_gb300 import roofline, workloads
    dev = torch.device("cuda", 0)
    G, B, d, dt = 8, 16, 128, torch.bfloat16
    L = 32  # layers moved per call (the pages' copies and swaps run over every layer)
    flush = torch.ones(128 * 1024 * 1024, dtype=torch.int32, device=dev)
    peak, _ = measured_hbm_peak()
    g = torch.Generator().manual_seed(0)
    line = {"workload": name}
    cpu = None
    clocks = ClockSampler(clocks_index)
    clocks.start()
    if name == "copy_blocks":
        wl = workloads.shared_prefix(device="cpu", cow=True)   # its 448 copy-on-write pairs and pool size
        pairs = wl.copy_pairs.to(dev)
        nb = wl.num_blocks
        kp = [torch.empty((nb, G, B, d), dtype=dt, device=dev) for _ in range(L)]
        vp = [torch.empty((nb, G, B, d), dtype=dt, device=dev) for _ in range(L)]
        ms = time_steps(lambda: pa.pa_copy_blocks(kp, vp, pairs), steps, warmup, flush)
        byt = roofline.copy_blocks_bytes(pairs.shape[0], L, B, G, d, 2)
        # the 7 samples of a prompt all copy its one partial block: reads repeat through L2
        nsrc = len(set(wl.copy_pairs[:, 0].tolist()))
        uniq = (nsrc + pairs.shape[0]) * L * roofline.kv_block_bytes(B, G, d, 2)
        line.update(desc=f"{pairs.shape[0]} CoW pairs ({nsrc} distinct sources) x {L} layers, bf16 blocks of "
                         f"16 x 8 heads x 128", bound="hbm",
                    unique_GBps=round(uniq / (ms * 1e-3) / 1e9, 1),
                    unique_frac_of_measured_peak=round(uniq / (ms * 1e-3) / 1e9 / peak, 4))
        P = int(pairs.shape[0])  # the oracle copies the same number of pairs within a compact pool
        kc = np.random.default_rng(0).integers(0, 1 << 16, (2 * P, G, B, d), dtype=np.uint16)
        cp = torch.stack([torch.arange(P), torch.arange(P, 2 * P)], 1)
        t = time.perf_counter()
        oracle.copy_blocks([kc], [kc.copy()], cp)
        cdt = time.perf_counter() - t
        cpu = {"value": round(roofline.copy_blocks_bytes(pairs.shape[0], 1, B, G, d, 2) / cdt / 1e9, 4),
               "unit": "GB/s", "cores": 1, "kind": "oracle", "seconds": round(cdt, 3),
               "sample": f"{pairs.shape[0]} pairs x 1 layer, numpy element copies"}
    elif name in ("swap_out", "swap_in"):
        nd, nh, P = 4096, 1024, 512
        dk = [torch.empty((nd, G, B, d), dtype=dt, device=dev) for _ in range(L)]
        dv = [torch.empty((nd, G, B, d), dtype=dt, device=dev) for _ in range(L)]
        hk = [torch.empty((nh, G, B, d), dtype=dt).pin_memory() for _ in range(L)]
        hv = [torch.empty((nh, G, B, d), dtype=dt).pin_memory() for _ in range(L)]
        src = torch.randperm(nd, generator=g)[:P]
        dst = torch.randperm(nh, generator=g)[:P]
        if name == "swap_out":
            pairs = torch.stack([src, dst], 1).to(dev)
            step = lambda: pa.pa_swap_blocks(hk, hv, dk, dv, pairs)  # noqa: E731
        else:
            pairs = torch.stack([dst, src], 1).to(dev)
            step = lambda: pa.pa_swap_blocks(dk, dv, hk, hv, pairs)  # noqa: E731
        ms = time_steps(step, steps, warmup, flush)
        byt = P * L * roofline.kv_block_bytes(B, G, d, 2)  # bytes moved across the host link
        # the same byte count as one contiguous copy over the same link, timed here
        dbuf = torch.empty(byt // 2, dtype=dt, device=dev)
        hbuf = torch.empty(byt // 2, dtype=dt).pin_memory()
        ref = (lambda: hbuf.copy_(dbuf, non_blocking=True)) if name == "swap_out" else \
            (lambda: dbuf.copy_(hbuf, non_blocking=True))
        ref_ms = time_steps(ref, steps, warmup, flush)
        line.update(desc=f"{P} blocks x {L} layers (K and V) {'device -> pinned host' if name == 'swap_out' else 'pinned host -> device'}, one launch",
                    bound="host link", contiguous_copy_GBps=round(byt / (ref_ms * 1e-3) / 1e9, 1),
                    frac_of_contiguous_copy=round(ref_ms / ms, 4))
    else:  # reshape (the benchmark step's 256 new tokens) or reshape_prefill (32 prompts x 1024 tokens)
        N = 256 if name == "reshape" else 32 * 1024
        nb = 100_000
        kc = torch.empty((nb, G, B, d), dtype=dt, device=dev)
        vc = torch.empty((nb, G, B, d), dtype=dt, device=dev)
        key = torch.randn((N, G, d), generator=g).to(dt).to(dev)
        val = torch.randn((N, G, d), generator=g).to(dt).to(dev)
        slots = torch.randperm(nb * B, generator=g)[:N].to(dev)
        ms = time_steps(lambda: pa.pa_reshape_and_cache(key, val, kc, vc, slots), steps, warmup, flush)
        byt = roofline.reshape_and_cache_bytes(N, G, d, 2)
        line.update(desc=f"{N} new tokens x 8 kv heads x 128 (bf16) into a 100k-block pool, random slots",
                    bound="hbm" if N > 1024 else "launch latency",
                    frac_of_measured_peak=round(byt / (ms * 1e-3) / 1e9 / peak, 4))
        n = min(N, 256)
        kh = np.zeros((64, G, B, d), np.uint16)
        t = time.perf_counter()
        oracle.reshape_and_cache(key[:n].cpu(), val[:n].cpu(), kh, kh.copy(), torch.arange(n, dtype=torch.int64))
        cdt = time.perf_counter() - t
        cpu = {"value": round(roofline.reshape_and_cache_bytes(n, G, d, 2) / cdt / 1e9, 4), "unit": "GB/s",
               "cores": 1, "kind": "oracle", "seconds": round(cdt, 3),
               "sample": f"{n} tokens, numpy element copies"}
    clk = clocks.stop()
    line.update(ms_per_step=round(ms, 5), algorithmic_GBps=round(byt / (ms * 1e-3) / 1e9, 1), bytes_per_step=byt,
                frac_of_nominal_peak=round(byt / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
                l2="512 MiB buffer read between timed steps", gpu_launches=steps,
                clocks=clk, device_errors=pa.pa_get_error())
    if cpu is not None and cpu_seconds:
        line["cpu_baseline"] = cpu
    return line


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e nominal (~8 TB/s), reported beside the measured copy peak

# The default run's other configurations, each a device-timed entry under "workloads"
# in the one JSON line (N = 1 only): the pages' workload shapes (OPT-13B MHA, the
# Llama-3.1-8B batch over E4M3 codes, 70B-shaped GQA-8 on short contexts, 64 prompts x 8
# samples sharing 2048-token prefixes, 70B-shaped 32K-128K contexts) and the CoW copies.
EXTRA_WORKLOADS = ("tiny", "opt13b", "llama8b_fp8", "llama70b_short", "shared", "shared_cascade", "shared_cow",
                   "shared_cow_cascade", "long70b_b16", "long70b_b32", "copy_blocks")


def build_workload(name, dev):
    """(workload, split, partition) for a named bench workload (a _nhd suffix stores the pools NHD)."""
    import torch
    from paged_kv_cache_04_gb300 import workloads
    import paged_kv_cache_04_gb300 as pa
    nhd = name.endswith("_nhd")
    base = name[:-4] if nhd else name
    split, T = False, None
    if base == "tiny":
        wl = workloads.tiny(device=dev)
    elif base == "opt13b":
        wl = workloads.opt13b(device=dev)
    elif base.startswith("shared"):
        # _x16: 32 prompts x 16 samples (64 query rows per group), _x32: 16 x 32 (128
        # rows), else 64 x 8 (32 rows); 512 sequences each
        shape = {"prompts": 32, "samples": 16} if "_x16" in base else (
            {"prompts": 16, "samples": 32} if "_x32" in base else {})
        wl = workloads.shared_prefix(device=dev, cow=base.startswith("shared_cow"), **shape)
        # set-up: the CoW copies and every appended token, once; a timed step then
        # repeats the copies and writes each sample's newest token before decoding
        if wl.copy_pairs.numel():
            pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], wl.copy_pairs)
        pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
        last = torch.tensor([int(wl.block_tables[s, (int(c) - 1) // wl.B]) * wl.B + (int(c) - 1) % wl.B
                             for s, c in enumerate(wl.context_lens.tolist())], dtype=torch.int64, device=dev)
        wl.slot_mapping = last
        wl.new_key, wl.new_value = wl.new_key[:wl.S].contiguous(), wl.new_value[:wl.S].contiguous()
    elif base in ("llama8b", "llama8b_fp8"):
        wl = workloads.llama8b(device=dev)
    elif base in ("llama8b_s2048", "llama8b_s2048_fp8"):  # the same shape and lengths, 2,048 sequences
        wl = workloads.llama8b(device=dev, S=2048, num_blocks=320_000)
    elif base in ("llama70b_short", "llama70b_short_fp8"):
        wl = workloads.llama70b_short(device=dev)
    elif base == "gemma_d256":
        wl = workloads.gemma_d256(device=dev)
    elif base.startswith("long70b"):
        wl = workloads.long70b(device=dev, B=32 if "b32" in base else 16)
        split, T = True, 512
    else:
        raise ValueError(f"unknown workload {name}")
    if base.endswith("fp8"):
        wl = workloads.to_fp8(wl)
    if nhd:
        wl = workloads.to_nhd(wl)
    torch.cuda.synchronize()
    return wl, split, T


def measure_workload(name, steps, warmup, cpu_seconds=None, clocks_index=0):
    """Device-timed steps of one named workload (single GPU): a dict with the step time,
    seqs/s, attended KV tokens/s, algorithmic GB/s against the measured and nominal HBM
    peaks, the attention call's own roofline, the clocks seen and (with cpu_seconds) the
    oracle on a bounded sample."""
    import torch
    import paged_kv_cache_04_gb300 as pa
    from paged_kv_cache_04_gb300 import _build, roofline
    _build.ensure_built()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if name in ("copy_blocks", "swap_out", "swap_in", "reshape", "reshape_prefill"):
        return measure_cache_workload(name, steps, warmup, cpu_seconds, clocks_index)
    wl, split, T = build_workload(name, dev)
    base = name[:-4] if name.endswith("_nhd") else name
    lay = wl.layout
    fp8 = base.endswith("fp8")
    cascade = base.endswith("cascade")
    ks, vs = wl.meta.get("k_scale", 1.0), wl.meta.get("v_scale", 1.0)
    if cascade:
        gs = torch.tensor(wl.meta["group_starts"], dtype=torch.int32, device=dev)
        pl = torch.tensor(wl.meta["prefix_lens"], dtype=torch.int32, device=dev)
        gmax = max(b - a for a, b in zip(wl.meta["group_starts"][:-1], wl.meta["group_starts"][1:]))
        pmax = max(wl.meta["prefix_lens"])
        T = 512
    out = torch.empty_like(wl.q)
    ws = None
    max_ctx = wl.max_context  # read once: it synchronises the device
    if cascade:
        ws = torch.empty(pa.pa_decode_cascade_workspace_bytes(wl.S, wl.H, wl.d, pmax, max_ctx, T),
                         dtype=torch.uint8, device=dev)
    if split:
        ws = torch.empty(pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, max_ctx, T),
                         dtype=torch.uint8, device=dev)
    # a buffer larger than L2, read between timed steps (a read leaves no dirty lines behind)
    flush = torch.ones(128 * 1024 * 1024, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    pairs = wl.copy_pairs if wl.copy_pairs is not None and wl.copy_pairs.numel() else None
    launches = 0

    def attend():
        if fp8:
            if split:
                pa.pa_decode_split_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                       wl.scale, ks, vs, max_ctx, T, ws, layout=lay)
            else:
                pa.pa_decode_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                                 ks, vs, layout=lay)
        elif cascade:
            pa.pa_decode_cascade(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                                 gs, pl, gmax, pmax, max_ctx, T, ws, layout=lay)
        elif split:
            pa.pa_decode_split(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                               max_ctx, T, ws, layout=lay)
        else:
            pa.pa_decode(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, layout=lay)

    # kernels one step launches: copies, cache write, then the attention call's launches
    attend_launches = 3 if cascade and max(wl.meta["prefix_lens"]) > 0 else (2 if split or cascade else 1)
    step_launches = attend_launches + (1 if wl.slot_mapping is not None else 0) + (1 if pairs is not None else 0)

    def step(ev=None):
        if pairs is not None:
            pa.pa_copy_blocks([wl.k_cache], [wl.v_cache], pairs)
        if wl.slot_mapping is not None:
            if fp8:
                pa.pa_reshape_and_cache_fp8(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping,
                                            ks, vs, layout=lay)
            else:
                pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping,
                                        layout=lay)
        if ev is not None:
            ev[0].record(stream)
        attend()
        if ev is not None:
            ev[1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(clocks_index)
    clocks.start()
    time.sleep(0.2)

    def timed(inner, cold=True):
        # inner: events around the attention call too (for its own roofline); they sit
        # between the cache write and the attention launch and stop that launch from
        # being scheduled early, so the step time comes from a loop without them.
        # cold: the flush read between steps (False: the L2 keeps what the last step left)
        nonlocal launches
        times = []
        # keep the GPU busy while the host queues every timed step, so no step waits on the host
        torch.cuda._sleep(int(2e6 * (2 + steps)))
        for _ in range(steps):
            if cold:
                flush.sum()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            ev[0].record(stream)
            step((ev[1], ev[2]) if inner else None)
            ev[3].record(stream)
            times.append(ev)
            launches += step_launches
        torch.cuda.synchronize()
        return (statistics.mean(e[0].elapsed_time(e[3]) for e in times),
                statistics.mean(e[1].elapsed_time(e[2]) for e in times) if inner else None)

    ms, _ = timed(False)
    _, att_ms = timed(True)
    # shared prefixes: also with the L2 left warm between steps (the prefix blocks a
    # step reads last may still be there for the next)
    warm_ms = timed(False, cold=False)[0] if base.startswith("shared") else None
    clk = clocks.stop()
    e = wl.q.element_size()
    ke = wl.k_cache.element_size()
    ctx = wl.context_lens.tolist()
    dec = (roofline.decode_bytes(ctx, wl.H, wl.G, wl.d, ke) - 2 * wl.S * wl.H * wl.d * ke
           + 2 * wl.S * wl.H * wl.d * e)  # K/V at the cache width, q and out at the query width
    extra = 0
    if wl.slot_mapping is not None:
        n = wl.slot_mapping.numel()
        extra += (roofline.reshape_and_cache_bytes(n, wl.G, wl.d, e) if not fp8
                  else 2 * n * wl.G * wl.d * (e + ke) + 8 * n)
    if pairs is not None:
        extra += roofline.copy_blocks_bytes(pairs.shape[0], 1, wl.B, wl.G, wl.d, e)
    unique = None
    if base.startswith("shared"):
        unique = wl.meta["unique_tokens"] * roofline.kv_bytes_per_token(1, wl.G, wl.d, e) + 2 * wl.S * wl.H * wl.d * e
    peak, peak_kind = measured_hbm_peak()
    gbps = (dec + extra) / (ms * 1e-3) / 1e9
    att_bytes = unique if unique is not None else dec
    att_gbps = att_bytes / (att_ms * 1e-3) / 1e9
    kernel = {"plain": "paged_decode_kernel (pa_decode)", "fp8": "paged_decode_kernel over E4M3 codes (pa_decode_fp8)",
              "split": "paged_decode_kernel split mode + lse_reduce (pa_decode_split, 2 launches)",
              "split_fp8": "paged_decode_kernel split mode over E4M3 codes + lse_reduce (pa_decode_split_fp8)",
              "cascade": "prefix pass + suffix pass + lse_reduce (pa_decode_cascade, 3 launches)"}[
        "cascade" if cascade else ("split_fp8" if split and fp8 else ("split" if split else ("fp8" if fp8 else "plain")))]
    line = {"workload": name, "seqs": wl.S, "q_heads": wl.H, "kv_heads": wl.G, "head_dim": wl.d, "block_size": wl.B,
            "cache_dtype": "e4m3" if fp8 else str(wl.k_cache.dtype).replace("torch.", ""), "layout": lay,
            "ms_per_step": round(ms, 5), "seqs_per_s": round(wl.S / (ms * 1e-3), 1),
            "kv_tokens_per_s": round(sum(ctx) / (ms * 1e-3), 1),
            "algorithmic_GBps": round(gbps, 1),
            "frac_of_measured_peak": round(gbps / peak, 4),
            "frac_of_nominal_peak": round(gbps / NOMINAL_HBM_GBS, 4),
            "bytes_per_step": dec + extra,
            "roofline": {"kernel": kernel, "bound": "hbm", "achieved": round(att_gbps, 1), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(att_gbps / peak, 4),
                         "frac_of_nominal": round(att_gbps / NOMINAL_HBM_GBS, 4), "traffic": None,
                         "algorithmic_bytes_per_launch": int(att_bytes), "avg_launch_ms": round(att_ms, 5),
                         "bytes_counted": "unique K/V (each shared prefix block once) + q + out" if unique is not None
                         else "K/V of every attended token + q + out"},
            "l2": "512 MiB buffer read between timed steps", "gpu_launches": launches, "clocks": clk,
            "device_errors": pa.pa_get_error()}
    if unique is not None:
        line["logical_GBps"] = line["algorithmic_GBps"]
        line["unique_GBps"] = round((unique + extra) / (ms * 1e-3) / 1e9, 1)
        line["unique_frac_of_measured_peak"] = round((unique + extra) / (ms * 1e-3) / 1e9 / peak, 4)
        line["copy_pairs"] = 0 if pairs is None else int(pairs.shape[0])
        line["warm_l2"] = {"ms_per_step": round(warm_ms, 5),
                           "unique_GBps": round((unique + extra) / (warm_ms * 1e-3) / 1e9, 1),
                           "unique_frac_of_measured_peak": round((unique + extra) / (warm_ms * 1e-3) / 1e9 / peak, 4),
                           "logical_GBps": round((dec + extra) / (warm_ms * 1e-3) / 1e9, 1),
                           "l2": "no flush between timed steps"}
    if cpu_seconds:
        line["cpu_baseline"] = decode_oracle_baseline(wl, cpu_seconds, fp8=fp8)
    return line


def run_workload(args):
    """One device-timed line for one of the other workload shapes (single GPU)."""
    line = measure_workload(args.workload, args.steps, args.warmup,
                            None if args.no_cpu_baseline else min(args.cpu_seconds, 5.0))
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """The step's kernels on a 64-sequence batch of the workload's shape (~0.6 GB of K/V per
    step, still larger than L2; ~1 GB pool), sized so that an ncu capture stays small."""
    import torch
    import paged_kv_cache_04_gb300 as pa
    from paged_kv_cache_04_gb300 import _build, workloads
    _build.ensure_built()
    dev = torch.device("cuda", 0)
    wl = workloads.llama8b(device=dev, S=64, num_blocks=16_000)
    if args.profile_fp8:
        wl = workloads.to_fp8(wl)
        torch.cuda.empty_cache()
    out = torch.empty_like(wl.q)
    ks, vs = wl.meta.get("k_scale", 1.0), wl.meta.get("v_scale", 1.0)
    for _ in range(args.warmup + args.steps):
        if args.profile_fp8:
            pa.pa_reshape_and_cache_fp8(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping, ks, vs)
            pa.pa_decode_fp8(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, ks, vs)
        else:
            pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
            pa.pa_decode(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    torch.cuda.synchronize()
    from paged_kv_cache_04_gb300 import roofline
    kv = roofline.decode_bytes(wl.context_lens.tolist(), wl.H, wl.G, wl.d, wl.k_cache.element_size())
    print(json.dumps({"profile_case": "llama8b S=64 pool 16000", "decode_bytes_per_launch": kv,
                      "source_sha256": kernel_source_sha(), "device_errors": pa.pa_get_error()}))


def run_cache_profile_case(args, name, dev):
    """The cache kernels on small cases for ncu. copy: the copy-on-write workload's 448
    pairs remapped into a compact pool of the 512 blocks they touch, 16 layers (537 MB
    of unique bytes per launch, 1.1 GB of pools); reshape: 32,768 new tokens into a
    20,000-block pool at random slots (268 MB per launch, 1.3 GB of pools)."""
    import torch
    import paged_kv_cache_04_gb300 as pa
    from paged_kv_cache_04_gb300 import roofline, workloads
    G, B, d, dt = 8, 16, 128, torch.bfloat16
    g = torch.Generator(device=dev).manual_seed(0)
    if name == "copy":
        L = 16
        pairs = workloads.shared_prefix(device="cpu", cow=True).copy_pairs
        blocks = sorted(set(pairs.flatten().tolist()))
        remap = {b: i for i, b in enumerate(blocks)}
        cp = torch.tensor([[remap[int(a)], remap[int(b)]] for a, b in pairs.tolist()], dtype=torch.int64,
                          device=dev)
        nb, P = len(blocks), int(pairs.shape[0])
        kp = [torch.randn((nb, G, B, d), generator=g, device=dev).to(dt) for _ in range(L)]
        vp = [torch.randn((nb, G, B, d), generator=g, device=dev).to(dt) for _ in range(L)]
        step = lambda: pa.pa_copy_blocks(kp, vp, cp)  # noqa: E731
        nsrc = len(set(pairs[:, 0].tolist()))
        info = {"pairs": P, "distinct_sources": nsrc, "layers": L, "pool_blocks": nb,
                "bytes_per_launch": roofline.copy_blocks_bytes(P, L, B, G, d, 2),
                "unique_bytes_per_launch": (nsrc + P) * L * roofline.kv_block_bytes(B, G, d, 2)}
    else:
        N, nb = 32 * 1024, 20_000
        kc = torch.empty((nb, G, B, d), dtype=dt, device=dev)
        vc = torch.empty((nb, G, B, d), dtype=dt, device=dev)
        key = torch.randn((N, G, d), generator=g, device=dev).to(dt)
        val = torch.randn((N, G, d), generator=g, device=dev).to(dt)
        slots = torch.randperm(nb * B, generator=g, device=dev)[:N]
        step = lambda: pa.pa_reshape_and_cache(key, val, kc, vc, slots)  # noqa: E731
        info = {"tokens": N, "pool_blocks": nb, "bytes_per_launch": roofline.reshape_and_cache_bytes(N, G, d, 2)}
    for _ in range(args.warmup + args.steps):
        step()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": name, **info, "device_errors": pa.pa_get_error()}))


def run_other_profile_case(args):
    """Small cases (K/V still larger than L2) of the split, shared-prefix and MHA paths, for ncu."""
    import torch
    import paged_kv_cache_04_gb300 as pa
    from paged_kv_cache_04_gb300 import _build, roofline, workloads
    _build.ensure_built()
    dev = torch.device("cuda", 0)
    name = args.profile_case
    if name in ("copy", "reshape"):
        run_cache_profile_case(args, name, dev)
        return
    if name == "split":
        wl = workloads.long70b(device=dev, S=2, lo=48_000, hi=64_000)
    elif name == "cascade":
        wl = workloads.shared_prefix(device=dev, prompts=32)
    elif name == "cascade_x16":  # 64 query rows per group: the tcgen05 prefix pass
        wl = workloads.shared_prefix(device=dev, prompts=16, samples=16)
    elif name == "g8":  # plain decode at group 8 (merge in rounds): ~0.57 GB of K/V, 4.4x the L2
        wl = workloads.llama70b_short(device=dev, S=64, num_blocks=16_000)
    else:
        wl = workloads.opt13b(device=dev)
    out = torch.empty_like(wl.q)
    mctx, T = wl.max_context, 512
    if name.startswith("cascade"):
        pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
        gs = torch.tensor(wl.meta["group_starts"], dtype=torch.int32, device=dev)
        pl = torch.tensor(wl.meta["prefix_lens"], dtype=torch.int32, device=dev)
        pmax = max(wl.meta["prefix_lens"])
        ws = torch.empty(pa.pa_decode_cascade_workspace_bytes(wl.S, wl.H, wl.d, pmax, mctx, T), dtype=torch.uint8,
                         device=dev)
    elif name == "split":
        ws = torch.empty(pa.pa_decode_split_workspace_bytes(wl.S, wl.H, wl.d, mctx, T), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup + args.steps):
        if name.startswith("cascade"):
            pa.pa_decode_cascade(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                                 gs, pl, wl.meta["samples"], pmax, mctx, T, ws)
        elif name == "split":
            pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
            pa.pa_decode_split(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                               mctx, T, ws)
        else:
            pa.pa_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
            pa.pa_decode(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    torch.cuda.synchronize()
    kv = roofline.decode_bytes(wl.context_lens.tolist(), wl.H, wl.G, wl.d, wl.k_cache.element_size())
    info = {"profile_case": name, "seqs": wl.S, "tokens": int(wl.context_lens.sum().item()),
            "decode_bytes_per_launch": kv, "device_errors": pa.pa_get_error()}
    if name.startswith("cascade"):
        info["unique_kv_tokens"] = wl.meta["unique_tokens"]
    print(json.dumps(info))


def main():
    args = parse()
    if args.record_traffic:
        record_traffic(args.record_traffic)
        return
    if args.profile or args.profile_fp8:
        run_profile_case(args)
        return
    if args.profile_case:
        run_other_profile_case(args)
        return
    if args.workload != "llama8b":
        run_workload(args)
        return
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world, local)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
