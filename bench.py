"""Benchmark: paged GQA decode attention on GB300.

One step = the whole hot path over one batch: append the new token of every
sequence into the paged pool and decode attention for every sequence
(paged_decode_step: the append fused into the decode kernel, then the
split-KV merge kernel).  The same step as two calls (paged_kv_append,
paged_decode_attention) is timed beside it.  The default workload is the 70B
long-context shape (n_q=64, n_kv=8, d_head=128, batch 16, every sequence at
32768 tokens: 2 GiB of bf16 K and V read per call), the largest of the
workloads; ``--workload`` picks another.

Prints one JSON line.  ``value`` is achieved KV-read bandwidth (algorithmic
bytes: K and V of every cached token + q + out, per step) in GB/s over the
device-timed region, summed over ranks; ``calls_per_s`` is decode calls per
second.  ``roofline`` is the decode kernel's event-timed fraction of the
measured copy peak; ``per_config`` gives the same fraction, the step time and
the parity against the oracle for each of the other workloads (tiny,
Llama3-8B, FP8 log-normal, shared prefix, 4-bit).  ``--impl reference`` times
the CPU oracle instead.

``--mode blocks`` instead measures the block-management kernels (copy-on-write
block copies, swap out / in over the CPU-GPU link) and ``--mode cascade``
the cascade decode over a shared prefix; each prints its own JSON line.

Run:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
N > 1 runs under torchrun as independent replicas (one per GPU, no
collective on the data path; a barrier and a max over ranks for timing).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged GQA decode: achieved KV-read GB/s vs GB300 HBM peak; attention calls/s"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="long_context_70b")
    p.add_argument("--partition-tokens", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--flush-l2", action="store_true", help="evict L2 between steps (512 MB written, 256 MB read)")
    p.add_argument("--no-per-config", action="store_true", help="skip the other workloads' per_config entries")
    p.add_argument("--kernel-seconds", type=float, default=1.0,
                   help="least duration of the per-kernel timing pass (the clock sampler runs through it)")
    p.add_argument("--config-seconds", type=float, default=0.4,
                   help="timed duration per workload of the per_config entries")
    p.add_argument("--mode", default="decode", choices=["decode", "blocks", "cascade", "prefill"])
    p.add_argument("--prefill-kv", default="bf16", choices=["bf16", "fp8"], help="--mode prefill: KV pool type")
    p.add_argument("--cascade-kv", default="bf16", choices=["bf16", "fp8"], help="--mode cascade: KV pool type")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; timing only)
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def init_dist(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def allreduce_max(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# byte accounting
# ---------------------------------------------------------------------------

def algorithmic_bytes(w) -> dict:
    """Bytes one decode call must move: K and V of every cached token of every
    sequence (logical), the same counted once per distinct slot (unique), q
    and out."""
    import numpy as np

    per_token = w.n_kv * w.kv_bytes_per_token_head  # K and V (4-bit: codes plus the value rows' scale and zero)
    logical_tokens = int(w.context_lens.astype(np.int64).sum())
    slots = set()
    if w.shared_prefix_tokens:
        for b in range(w.batch):
            C = int(w.context_lens[b])
            nb = (C + w.block_size - 1) // w.block_size
            for j in range(nb):
                n = min(w.block_size, C - j * w.block_size)
                slots.update(int(w.block_tables[b, j]) * w.block_size + o for o in range(n))
        unique_tokens = len(slots)
    else:
        unique_tokens = logical_tokens
    qo = 2 * w.batch * w.n_q * w.d_head * 2
    return {
        "kv_logical": logical_tokens * per_token,
        "kv_unique": unique_tokens * per_token,
        "q_out": qo,
        "logical": logical_tokens * per_token + qo,
        "unique": unique_tokens * per_token + qo,
        "flops": 4 * w.n_q * w.d_head * logical_tokens,
    }


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, no MEASURED_PEAKS.json)"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for rel in ("gqa_decode_attention_paged_gb300/csrc/decode.cu",
                "gqa_decode_attention_paged_gb300/csrc/pkv_internal.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, sha: str):
    """dram bytes per decode launch from profiles/traffic.txt, if taken on this source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None, None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == "decode_kernel" and parts[1] == workload:
            if parts[2] == sha:
                return float(parts[3]), " ".join(parts[4:])
    return None, None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, "t_" + which, time.time())

    def stop(self):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        for t, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((t, float(parts[0]), float(parts[1]), float(parts[2]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if self.t_start and self.t_stop and self.t_start <= r[0] <= self.t_stop]
        used = inside
        note = "samples taken during the sampled window"
        if not used:  # region shorter than the sampling period: nearest samples after its start
            used = sorted(rows, key=lambda r: abs(r[0] - (self.t_stop or r[0])))[:2]
            note = "timed region shorter than the 100 ms sampling period; nearest samples"
        reasons = sorted({self.NAMES[i] for r in used for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "power_w_max": max(r[3] for r in used), "reasons": reasons, "samples": len(used),
                "note": note}


def gpu_id_for(device_index: int) -> str:
    import torch

    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        if u and not u.startswith("GPU-"):
            u = "GPU-" + u
        return u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device_index] if vis else str(device_index)


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_setup(w):
    import oracle

    dt = {"bf16": oracle.BF16, "fp8": oracle.E4M3, "int4": oracle.INT4}[w.dtype]
    m = oracle.PoolMirror(w.num_blocks, w.block_size, w.n_kv, w.d_head, dt, w.k_scale, w.v_scale, w.k_zero)
    m.append(w.fill_k, w.fill_v, w.fill_slots)
    return m


def oracle_step(m, w, seqs):
    """The oracle's step on the sequences `seqs`: append their new tokens, decode them."""
    import numpy as np

    idx = np.asarray(seqs)
    m.append(w.step_k[idx], w.step_v[idx], w.step_slots[idx])
    return m.decode(w.q[idx], w.block_tables[idx], w.context_lens[idx], w.scale)


def _bytes_per_sequence(w) -> list:
    """Bytes one sequence's decode must move, as algorithmic_bytes counts them:
    its cached K and V (4-bit: codes plus the value rows' scale and zero), q and out."""
    per_token = w.n_kv * w.kv_bytes_per_token_head
    return [int(c) * per_token + 2 * w.n_q * w.d_head * 2 for c in w.context_lens]


def time_oracle(w, m, budget_s: float, max_reps: int = 20000):
    """Time oracle steps over rotating single sequences until budget_s; returns
    (GB/s, seconds, sequences done, threads)."""
    import numpy as np

    import oracle

    per_seq = _bytes_per_sequence(w)
    done_bytes, n, t0 = 0, 0, time.perf_counter()
    b = 0
    while n < max_reps:
        oracle_step(m, w, [b])
        done_bytes += per_seq[b]
        n += 1
        b = (b + 1) % w.batch
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return done_bytes / dt / 1e9, dt, n, oracle.hardware_threads(), np.mean(per_seq)


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import workloads as wl

    w = wl.NAMED[args.workload]()
    m = oracle_setup(w)
    # Each step decodes one sequence (rotating); sized so the run ends in minutes.
    times = []
    per_seq = _bytes_per_sequence(w)
    total_bytes = 0
    budget = 150.0
    t_run = time.perf_counter()
    steps = args.steps
    for i in range(args.warmup + args.steps):
        if time.perf_counter() - t_run > budget and i >= args.warmup + 1:
            steps = i - args.warmup
            break
        b = i % w.batch
        t0 = time.perf_counter()
        oracle_step(m, w, [b])
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            total_bytes += per_seq[b]
    import oracle

    secs = sum(times)
    gbs = total_bytes / secs / 1e9 if secs > 0 else 0.0
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": len(times),
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, len(times)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(w.describe(), parallelism="replicas"),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": oracle.hardware_threads(), "kind": "oracle",
                         "sample": f"one sequence (all {w.n_q} heads) per step, rotating over the "
                                   f"{w.batch} sequences of the workload; steps requested {args.steps}, "
                                   f"run {len(times)} within a {budget:.0f} s budget"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


class L2Flush:
    """Evicts L2 between timed calls: writes a 512 MB buffer (larger than the
    129 MB L2), then reads a separate 256 MB one, so that the timed call
    starts with a cold L2 that holds no dirty lines of the flush (their write
    back would otherwise land inside the timed call)."""

    def __init__(self, device):
        import torch

        self.w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
        self.r = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.fill_(1)
        self.r.max()


class DecodeRig:
    """One workload's pool and step inputs on the device, and its step: the
    fused append + decode call (paged_decode_step), or for 4-bit pools the
    append then the decode."""

    def __init__(self, w, device, partition_tokens: int = 0):
        import numpy as np
        import torch

        import gqa_decode_attention_paged_gb300 as pkv

        self.pkv, self.w, self.device = pkv, w, device
        dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(device).view(dt)  # noqa: E731
        dt = {"bf16": pkv.BF16, "fp8": pkv.FP8_E4M3, "int4": pkv.INT4}[w.dtype]
        self.pool = pkv.kv_pool_create(w.num_blocks, w.block_size, w.n_kv, w.d_head, dt)
        if w.dtype == "fp8":
            self.pool.set_fp8_scales(w.k_scale, w.v_scale)
        if w.dtype == "int4":
            self.pool.set_int4_key_params(w.k_scale, w.k_zero)
        if partition_tokens:
            self.pool.set_partition_tokens(partition_tokens)
        self.pool.reserve_workspace(w.batch, w.n_q, w.max_blocks_per_seq)
        T = w.fill_slots.shape[0]
        for s in range(0, T, 1 << 20):
            e = min(T, s + (1 << 20))
            pkv.paged_kv_append(self.pool, dev(w.fill_k[s:e].view(np.int16), torch.bfloat16),
                                dev(w.fill_v[s:e].view(np.int16), torch.bfloat16), dev(w.fill_slots[s:e], torch.int64))
        self.k_new = dev(w.step_k.view(np.int16), torch.bfloat16)
        self.v_new = dev(w.step_v.view(np.int16), torch.bfloat16)
        self.slots = dev(w.step_slots, torch.int64)
        self.q = dev(w.q.view(np.int16), torch.bfloat16)
        self.tables = dev(w.block_tables, torch.int32)
        self.lens = dev(w.context_lens, torch.int32)
        self.out = torch.empty_like(self.q)
        self.stream = torch.cuda.current_stream()
        self.scale = float(w.scale)
        torch.cuda.synchronize()

    def step(self):
        """One pass of the hot path: append every sequence's new token, decode."""
        pkv, p = self.pkv, self.pool
        if self.w.dtype == "int4":  # no fused step for 4-bit pools: append, then decode
            pkv.paged_kv_append(p, self.k_new, self.v_new, self.slots, self.stream)
            pkv.paged_decode_attention(p, self.q, self.tables, self.lens, self.scale, self.out, self.stream)
        else:
            pkv.paged_decode_step(p, self.q, self.k_new, self.v_new, self.tables, self.lens, self.scale, self.out,
                                  self.stream)

    def step_two_calls(self):
        pkv, p = self.pkv, self.pool
        pkv.paged_kv_append(p, self.k_new, self.v_new, self.slots, self.stream)
        pkv.paged_decode_attention(p, self.q, self.tables, self.lens, self.scale, self.out, self.stream)

    def kernel_pass(self, n: int, flush=None) -> dict:
        """n steps with a CUDA event pair recorded by the library around each
        of its launches on the launching stream; per-kernel averages."""
        import torch

        self.pool.timing_read(reset=True)
        self.pool.timing_enable(True)
        for _ in range(n):
            if flush is not None:
                flush()
            self.step()
        torch.cuda.synchronize()
        self.pool.timing_enable(False)
        tm = self.pool.timing_read(reset=True)
        return {"decode_ms": tm["decode_ms"] / max(1, tm["timed_decode"]),
                "merge_ms": tm["merge_ms"] / max(1, tm["timed_merge"]),
                "append_ms": tm["append_ms"] / max(1, tm["timed_append"]), "steps": n}

    def timed_steps(self, n: int, flush=None) -> float:
        """ms per step: events around n back-to-back steps, or with a flush,
        an event pair around each step (the flush outside it)."""
        import torch

        if flush is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for _ in range(n):
                self.step()
            e1.record(self.stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush()
            a.record(self.stream)
            self.step()
            b.record(self.stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / n

    def close(self):
        import torch

        self.pool.close()
        for name in ("k_new", "v_new", "slots", "q", "tables", "lens", "out"):
            setattr(self, name, None)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def parity_vs_oracle(w, got_bits) -> dict:
    """The oracle's step on the whole batch against the GPU output (bf16
    patterns, [B][n_q][d]); the tolerances of the parity tests."""
    import numpy as np

    import workloads as wl

    m = oracle_setup(w)
    ref = oracle_step(m, w, list(range(w.batch)))
    got = wl.bf16_bits_to_f32(got_bits).reshape(ref.shape).astype(np.float64)
    err = np.abs(got - ref)
    return {"max_abs": float(err.max()), "mean_abs": float(err.mean()), "tol_max_abs": 1e-2, "tol_mean_abs": 1e-3,
            "ok": bool(np.isfinite(got).all() and err.max() <= 1e-2 and err.mean() <= 1e-3),
            "sample": f"every output of the batch ({w.batch} sequences x {w.n_q} heads x {w.d_head})"}, m


def out_bits(t):
    import numpy as np
    import torch

    return t.view(torch.int16).cpu().numpy().view(np.uint16)


# Workloads whose KV is under ~4x L2 are timed with L2 flushed between calls.
FLUSHED = {"tiny", "shared_prefix"}
PER_CONFIG = ["long_context_70b", "llama3_8b", "fp8_lognormal", "shared_prefix", "int4_llama3", "tiny"]


def measure_config(name: str, device, warmup: int, seconds: float, peak: float, sha: str) -> dict:
    """One workload's decode-kernel roofline fraction, step time and parity
    against the oracle (a per_config entry of the bench line)."""
    import workloads as wl

    w = wl.NAMED[name]()
    acct = algorithmic_bytes(w)
    shared = w.shared_prefix_tokens > 0
    step_bytes = acct["unique"] if shared else acct["logical"]
    flush = L2Flush(device) if name in FLUSHED else None
    rig = DecodeRig(w, device)
    try:
        for _ in range(max(3, warmup)):
            if flush is not None:
                flush()
            rig.step()
        probe_ms = rig.timed_steps(5, flush)
        n = int(max(50, min(2000 if flush is not None else 20000, seconds * 1e3 / max(probe_ms, 1e-3))))
        step_ms = rig.timed_steps(n, flush)
        kt = rig.kernel_pass(n, flush)
        assert rig.pool.get_error() == 0, f"device error on {name}"
        got = out_bits(rig.out)
    finally:
        rig.close()
        del flush
    parity, _ = parity_vs_oracle(w, got)
    traffic, traffic_note = ncu_traffic(w.name, sha)
    achieved = step_bytes / (kt["decode_ms"] / 1e3) / 1e9
    return {
        "workload": w.name, "kv_dtype": w.dtype, "bytes_per_launch": step_bytes,
        "bytes_basis": "unique KV slots" if shared else "logical KV",
        "l2": "flushed before every step (512 MB written, 256 MB read)" if name in FLUSHED else
              f"inputs larger than L2 ({acct['kv_unique'] / 1e6:.0f} MB of KV per call)",
        "decode_kernel_ms": kt["decode_ms"], "merge_kernel_ms": kt["merge_ms"],
        "achieved_gbs": achieved, "frac": achieved / peak, "step_ms": step_ms,
        "step_gbs": step_bytes / (step_ms / 1e3) / 1e9, "steps_timed": n,
        "traffic": traffic, "traffic_source": traffic_note, "parity": parity,
    }


def run_ours(args):
    import numpy as np
    import torch

    import gqa_decode_attention_paged_gb300 as pkv
    import workloads as wl

    rank, local_rank, world = dist_env()
    if world != args.gpus and world > 1:
        print(f"warning: WORLD_SIZE={world} but --gpus={args.gpus}", file=sys.stderr)
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    init_dist(world, "nccl")

    w = wl.NAMED[args.workload]()
    acct = algorithmic_bytes(w)
    use_unique = w.shared_prefix_tokens > 0
    step_bytes = acct["unique"] if use_unique else acct["logical"]
    rig = DecodeRig(w, device, args.partition_tokens)
    pool, stream = rig.pool, rig.stream
    flush = L2Flush(device) if args.flush_l2 else None

    for _ in range(args.warmup):
        if flush is not None:
            flush()
        rig.step()
    torch.cuda.synchronize()
    assert pool.get_error() == 0, "device error during warm-up"

    # ---- device-timed region: exactly K steps ----
    sampler = ClockSampler(gpu_id_for(local_rank)) if rank == 0 else None
    if sampler:
        sampler.start()
    pool.timing_read(reset=True)  # zero the launch counters; no per-kernel events in this region
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("start")
    t_wall0 = time.perf_counter()
    step_ms_avg = rig.timed_steps(args.steps, flush)
    elapsed_ms = step_ms_avg * args.steps
    t_region = time.perf_counter() - t_wall0
    if sampler:
        sampler.mark("region_end")
    barrier(world)
    launches = int(pool.timing_read(reset=True)["launches"])
    assert pool.get_error() == 0, "device error in the timed region"

    # ---- kernel durations: the same step again, for at least --kernel-seconds,
    # with a CUDA event pair recorded by the library around each of its launches
    # on the launching stream; the clock sampler keeps running through it ----
    n_k = int(max(args.steps, min(3000 if flush is not None else 50000,
                                  args.kernel_seconds * 1e3 / max(step_ms_avg, 1e-3))))
    kt = rig.kernel_pass(n_k, flush)
    if sampler:
        sampler.mark("stop")
        sampler.stop()
    max_ms = allreduce_max(elapsed_ms, world, device)
    total_bytes = allreduce_sum(step_bytes * args.steps, world, device)

    # the same step as two calls (paged_kv_append, then paged_decode_attention), for comparison
    n2 = max(3, min(n_k, 1000))
    for _ in range(3):
        rig.step_two_calls()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(n2):
        rig.step_two_calls()
    ev1.record(stream)
    torch.cuda.synchronize()
    two_call_ms = ev0.elapsed_time(ev1) / n2
    value = total_bytes / (max_ms / 1e3) / 1e9
    calls = allreduce_sum(args.steps, world, device) / (max_ms / 1e3)

    # ---- end to end through the public API, host buffers ----
    e2e = None
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        h_q, h_k, h_v = (pin(x.view(np.int16)).view(torch.bfloat16) for x in (w.q, w.step_k, w.step_v))
        h_t, h_c = pin(w.block_tables), pin(w.context_lens)
        h_out = torch.empty(tuple(rig.q.shape), dtype=torch.bfloat16).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in (h_q, h_k, h_v, h_t, h_c))
        d2h = h_out.numel() * h_out.element_size()

        # the public host-buffer step on fixed pinned buffers (reads them in, appends, decodes,
        # writes the output back, synchronises)
        e2e_step = pkv.HostStep(pool, h_q, h_k, h_v, h_t, h_c, float(w.scale), h_out, stream)

        for _ in range(max(3, min(args.warmup, 10))):
            e2e_step()
        n_e2e = int(max(args.steps, min(20000, 0.5e3 / max(step_ms_avg, 1e-3))))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        e2e_s = allreduce_max(time.perf_counter() - t0, world, device)
        e2e_total = allreduce_sum(step_bytes * n_e2e, world, device)
        e2e = {"value": e2e_total / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": n_e2e, "ms_per_step": 1e3 * e2e_s / n_e2e,
               "calls_per_s": allreduce_sum(n_e2e, world, device) / e2e_s,
               "call": "HostStep: paged_decode_step_host on fixed pinned host inputs and output"}
    got_main = out_bits(rig.out)
    rig.close()
    del flush

    if rank != 0:
        return 0

    peak, peak_note = measured_peaks()
    sha = kernel_source_sha()
    # ---- the other workloads: decode-kernel fraction and parity, one at a time ----
    per_config = {}
    if not args.no_per_config:
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            per_config[name] = measure_config(name, device, args.warmup, args.config_seconds, peak, sha)

    # ---- the CPU-baseline leg: the oracle (test infrastructure) runs this
    # step on the host; its output of the full batch also gives the parity
    # figures for this very launch configuration, then it is timed ----
    cpu, parity = None, None
    if not args.no_cpu_baseline:
        parity, m = parity_vs_oracle(w, got_main)
        gbs, secs, nseq, threads, _ = time_oracle(w, m, budget_s=12.0)
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{nseq} single-sequence oracle steps (append + decode, all {w.n_q} heads, "
                         f"fp64, {threads} threads) rotating over the workload's sequences, {secs:.1f} s"}

    dec_ms = kt["decode_ms"]
    traffic, traffic_note = ncu_traffic(w.name, sha)
    achieved = step_bytes / (dec_ms / 1e3) / 1e9
    clocks = sampler.summary() if sampler else None
    if clocks is not None:
        clocks["window"] = (f"the timed region ({args.steps} steps, {t_region * 1e3:.1f} ms) and the kernel-timing "
                            f"pass right after it ({n_k} steps of the same workload)")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "calls_per_s": calls,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": max_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": dict(w.describe(), parallelism="replicas" if world > 1 else "single GPU",
                       bytes_per_step=step_bytes, bytes_basis="unique KV slots" if use_unique else "logical KV",
                       kv_bytes_logical=acct["kv_logical"], kv_bytes_unique=acct["kv_unique"],
                       l2=("flushed between steps (512 MB written, then 256 MB read)" if args.flush_l2 else
                           f"inputs larger than L2: {acct['kv_unique'] / 1e6:.0f} MB of KV per call vs 129 MB L2"),
                       work_split=(f"slices of {args.partition_tokens} tokens" if args.partition_tokens
                                   else "one equal slice of the batch's blocks per resident warp")),
        "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "bytes_per_launch": step_bytes, "avg_launch_ms": dec_ms, "peak_source": peak_note,
                     "traffic_source": traffic_note, "kernel_source_sha": sha},
        "kernels_ms_avg": {"decode_kernel": dec_ms, "merge_kernel": kt["merge_ms"]},
        "step_call": ("paged_kv_append, then paged_decode_attention (decode and split-KV merge kernels)"
                      if w.dtype == "int4" else
                      "paged_decode_step (the append fused into the decode kernel, then the split-KV merge "
                      "kernel: two launches)"),
        "two_call_step_ms": two_call_ms,
        "step_frac_of_peak": value / world / peak,
        "gpu_launches": launches,
        "kernel_timing_steps": n_k,
        "clocks": clocks,
        "parity": parity,
        "per_config": per_config,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "flops_per_step": acct["flops"],
    }
    if use_unique:
        line["effective_logical_gbs"] = acct["logical"] * args.steps * world / (max_ms / 1e3) / 1e9
    print(json.dumps(line))
    return 0


def _timed(fn, reps: int, warmup: int, stream, flush=None) -> float:
    """ms per call of fn(): CUDA events around `reps` back-to-back calls, or,
    with a `flush` buffer, an event pair around each call with the buffer
    written (evicting L2) before it."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if flush is not None:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in evs:
            flush()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / reps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_blocks(args):
    """Copy-on-write block copies and swaps on a Llama3-8B-shaped pool
    (n_kv 8, d_head 128, bf16: 64 KiB per block, K and V)."""
    import numpy as np
    import torch

    import gqa_decode_attention_paged_gb300 as pkv

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    NB, n = 8192, 2048  # 512 MiB pool; 2048 blocks = 128 MiB per direction
    pool = pkv.kv_pool_create(NB, 16, 8, 128, pkv.BF16)
    bb = pkv.kv_block_bytes(pool)
    g = torch.Generator(device="cuda").manual_seed(5)
    kview, vview = pool.k_view(), pool.v_view()  # strided views into the pool's (block, head) entries
    kview.copy_(torch.randint(0, 256, tuple(kview.shape), dtype=torch.uint8, device="cuda", generator=g))
    vview.copy_(torch.randint(0, 256, tuple(vview.shape), dtype=torch.uint8, device="cuda", generator=g))
    perm = np.random.default_rng(3).permutation(NB).astype(np.int32)
    src = torch.from_numpy(perm[:n]).cuda()
    dst = torch.from_numpy(perm[n:2 * n]).cuda()
    reps = max(3, min(args.steps, 200))
    warm = max(3, args.warmup)
    copy_ms = _timed(lambda: pkv.kv_block_copy(pool, src, dst, stream), reps, warm, stream)
    # exact: every destination block equals its source, K and V
    kv, vv = kview.reshape(NB, -1), vview.reshape(NB, -1)  # copies: read after the block copies ran
    copy_ok = bool(torch.equal(kv[dst.long()], kv[src.long()]) and torch.equal(vv[dst.long()], vv[src.long()]))
    copy_bytes = 2 * n * 2 * bb  # read + write, K and V
    host = torch.empty(n * 2 * bb, dtype=torch.uint8).pin_memory()
    out_ms = _timed(lambda: pkv.kv_swap_out(pool, src, host, stream), reps // 4 + 3, warm, stream)
    img_ok = bool(torch.equal(host.view(n, 2, bb)[:, 0].cuda(), kv[src.long()])
                  and torch.equal(host.view(n, 2, bb)[:, 1].cuda(), vv[src.long()]))
    in_ms = _timed(lambda: pkv.kv_swap_in(pool, host, dst, stream), reps // 4 + 3, warm, stream)
    swap_bytes = n * 2 * bb
    # the link's copy engine on the same bytes, for reference
    dev_buf = torch.empty(swap_bytes, dtype=torch.uint8, device="cuda")
    d2h_ms = _timed(lambda: host.copy_(dev_buf, non_blocking=True), reps // 4 + 3, warm, stream)
    h2d_ms = _timed(lambda: dev_buf.copy_(host, non_blocking=True), reps // 4 + 3, warm, stream)
    assert pool.get_error() == 0
    peak, peak_note = measured_peaks()
    gbs = lambda b, ms: b / (ms / 1e3) / 1e9  # noqa: E731
    line = {
        "metric": "paged KV block management: copy-on-write block copy GB/s (read+write) vs HBM peak; "
                  "swap out/in GB/s vs the copy engine on the same link",
        "mode": "blocks",
        "value": gbs(copy_bytes, copy_ms),
        "unit": "GB/s",
        "higher_is_better": True,
        "dtype": "bytes",
        "data": "synthetic",
        "config": {"workload": "llama3_8b_pool_blocks", "num_blocks": NB, "n_kv": 8, "d_head": 128,
                   "kv_dtype": "bf16", "block_bytes_kv": 2 * bb, "blocks_moved": n},
        "roofline": {"bound": "hbm", "kernel": "block_move_kernel<copy>", "achieved": gbs(copy_bytes, copy_ms),
                     "peak": peak, "unit": "GB/s", "frac": gbs(copy_bytes, copy_ms) / peak,
                     "peak_source": peak_note, "bytes_per_launch": copy_bytes, "avg_launch_ms": copy_ms},
        "swap_out": {"value": gbs(swap_bytes, out_ms), "unit": "GB/s", "ms": out_ms,
                     "copy_engine_d2h_gbs": gbs(swap_bytes, d2h_ms), "frac_of_copy_engine": d2h_ms / out_ms},
        "swap_in": {"value": gbs(swap_bytes, in_ms), "unit": "GB/s", "ms": in_ms,
                    "copy_engine_h2d_gbs": gbs(swap_bytes, h2d_ms), "frac_of_copy_engine": h2d_ms / in_ms},
        "parity": {"copy_bit_exact": copy_ok, "swap_out_bit_exact": img_ok, "ok": copy_ok and img_ok},
        "gpu_launches": int(pool.timing_read(reset=True)["block_launches"]),
    }
    print(json.dumps(line), flush=True)
    pool.close()
    return 0


def run_cascade(args):
    """Cascade decode (shared prefix read once) against plain decode on the
    shared-prefix workload; bytes counted on unique KV slots."""
    import numpy as np
    import torch

    import gqa_decode_attention_paged_gb300 as pkv
    import workloads as wl

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    # the named workload if it has a shared prefix (shared_prefix, shared_prefix_long), else shared_prefix
    w = wl.NAMED[args.workload]() if args.workload in wl.NAMED else None
    if w is None or not w.shared_prefix_tokens:
        w = wl.shared_prefix()
    if args.cascade_kv == "fp8":  # the same lengths and shared prefix on an FP8 E4M3 pool
        w = wl.build(w.name + "_fp8", w.n_q, w.n_kv, w.d_head, w.context_lens, dtype="fp8", seed=w.seed,
                     shared_prefix_tokens=w.shared_prefix_tokens, max_blocks_per_seq=w.max_blocks_per_seq)
    acct = algorithmic_bytes(w)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).cuda().view(dt)  # noqa: E731
    pool = pkv.kv_pool_create(w.num_blocks, w.block_size, w.n_kv, w.d_head,
                              pkv.FP8_E4M3 if args.cascade_kv == "fp8" else pkv.BF16)
    if args.cascade_kv == "fp8":
        pool.set_fp8_scales(w.k_scale, w.v_scale)
    pkv.paged_kv_append(pool, dev(w.fill_k.view(np.int16), torch.bfloat16), dev(w.fill_v.view(np.int16), torch.bfloat16),
                        dev(w.fill_slots, torch.int64))
    pkv.paged_kv_append(pool, dev(w.step_k.view(np.int16), torch.bfloat16), dev(w.step_v.view(np.int16), torch.bfloat16),
                        dev(w.step_slots, torch.int64))
    q = dev(w.q.view(np.int16), torch.bfloat16)
    tables = dev(w.block_tables, torch.int32)
    lens = dev(w.context_lens, torch.int32)
    n_pre = w.shared_prefix_tokens // 16
    # what the library's automatic mode picks for this prefix and batch, then the cascade forced
    pool.timing_read(reset=True)
    pkv.paged_decode_attention_prefix(pool, q, dev(w.block_tables[0, :n_pre], torch.int32), tables, lens,
                                      float(w.scale), torch.empty_like(q), stream)
    torch.cuda.synchronize()
    auto_cascade = pool.timing_read(reset=True)["prefix_launches"] > 0
    pool.set_cascade_mode(pkv.CASCADE_ALWAYS)
    pre = dev(w.block_tables[0, :n_pre], torch.int32)
    out_c, out_p = torch.empty_like(q), torch.empty_like(q)
    reps, warm = max(3, min(args.steps, 500)), max(3, args.warmup)
    flush = L2Flush("cuda") if args.flush_l2 else None
    casc_ms = _timed(lambda: pkv.paged_decode_attention_prefix(pool, q, pre, tables, lens, float(w.scale), out_c, stream),
                     reps, warm, stream, flush)
    plain_ms = _timed(lambda: pkv.paged_decode_attention(pool, q, tables, lens, float(w.scale), out_p, stream),
                      reps, warm, stream, flush)
    # the two paths on the same inputs (each is checked against the oracle by the tests)
    err = (out_c.float() - out_p.float()).abs().cpu().numpy()
    assert pool.get_error() == 0
    peak, peak_note = measured_peaks()
    gbs = acct["unique"] / (casc_ms / 1e3) / 1e9
    line = {
        "metric": "cascade decode over a shared prefix: unique KV-read GB/s vs GB300 HBM peak",
        "mode": "cascade",
        "value": gbs,
        "unit": "GB/s",
        "higher_is_better": True,
        "ms_per_call": casc_ms,
        "plain_decode_ms_per_call": plain_ms,
        "speedup_vs_plain": plain_ms / casc_ms,
        "auto_mode_picks": "cascade" if auto_cascade else "plain decode",
        "dtype": "f32",
        "data": "synthetic",
        "config": dict(w.describe(), bytes_basis="unique KV slots", kv_bytes_unique=acct["kv_unique"],
                       kv_bytes_logical=acct["kv_logical"],
                       l2=("flushed before each timed call (512 MB written, 256 MB read)" if flush is not None else
                           "not flushed: back-to-back calls")),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_source": peak_note},
        "agreement_with_plain_decode": {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
                                        "ok": bool(err.max() <= 1e-2 and err.mean() <= 1e-3)},
    }
    print(json.dumps(line), flush=True)
    pool.close()
    return 0


def run_prefill(args):
    """Chunked prefill attention: a 512-token chunk for each of the Llama3-8B
    batch's 64 sequences (caches of 1024..2048 tokens, the chunk being their
    last 512 positions), causal over the cache.  Tensor-bound: reported in
    attention TFLOP/s (4 x n_q x d_head per query token and visible key)."""
    import numpy as np
    import torch

    import gqa_decode_attention_paged_gb300 as pkv
    import workloads as wl

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    w = wl.llama3_8b()
    if args.prefill_kv == "fp8":  # the same lengths on an FP8 E4M3 pool
        w = wl.build("llama3_8b_fp8_b64", 32, 8, 128, w.context_lens, dtype="fp8", seed=12)
    T = 512
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).cuda().view(dt)  # noqa: E731
    pool = pkv.kv_pool_create(w.num_blocks, w.block_size, w.n_kv, w.d_head,
                              pkv.FP8_E4M3 if args.prefill_kv == "fp8" else pkv.BF16)
    if args.prefill_kv == "fp8":
        pool.set_fp8_scales(w.k_scale, w.v_scale)
    pkv.paged_kv_append(pool, dev(w.fill_k.view(np.int16), torch.bfloat16), dev(w.fill_v.view(np.int16), torch.bfloat16),
                        dev(w.fill_slots, torch.int64))
    pkv.paged_kv_append(pool, dev(w.step_k.view(np.int16), torch.bfloat16), dev(w.step_v.view(np.int16), torch.bfloat16),
                        dev(w.step_slots, torch.int64))
    rng = np.random.default_rng(11)
    q_bits = wl.f32_to_bf16_bits(rng.normal(size=(w.batch * T, w.n_q, w.d_head)).astype(np.float32))
    q = dev(q_bits.view(np.int16), torch.bfloat16)
    indptr = dev(np.arange(0, w.batch * T + 1, T, dtype=np.int32), torch.int32)
    tables = dev(w.block_tables, torch.int32)
    lens = dev(w.context_lens, torch.int32)
    out = torch.empty_like(q)
    reps, warm = max(3, min(args.steps, 50)), max(3, args.warmup)
    ms = _timed(lambda: pkv.paged_prefill_attention(pool, q, indptr, tables, lens, float(w.scale), out, stream),
                reps, warm, stream)
    assert pool.get_error() == 0
    C = w.context_lens.astype(np.int64)
    keys = int(sum(int(c) * T - T * (T - 1) // 2 for c in C))  # sum over chunk tokens of visible keys
    flops = 4 * w.n_q * w.d_head * keys
    tflops = flops / (ms / 1e3) / 1e12
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(peaks.get("bf16_tflops", 1900.0))
    line = {
        "metric": "chunked prefill attention over the paged cache: attention TFLOP/s vs GB300 bf16 tensor peak",
        "mode": "prefill",
        "value": tflops,
        "unit": "TFLOP/s",
        "higher_is_better": True,
        "ms_per_call": ms,
        "dtype": ("E4M3 K/V widened to f16, f16 q and P, f32 accumulate" if args.prefill_kv == "fp8"
                  else "bf16 in, f32 accumulate"),
        "data": "synthetic",
        "config": dict(w.describe(), chunk_tokens=T, query_rows=w.batch * T, visible_keys=keys),
        "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel", "achieved": tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": tflops / peak,
                     "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops: cuBLAS burst)" if peaks
                     else "fallback"},
    }
    print(json.dumps(line), flush=True)
    pool.close()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "prefill":
        return run_prefill(args)
    if args.mode == "blocks":
        return run_blocks(args)
    if args.mode == "cascade":
        return run_cascade(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
