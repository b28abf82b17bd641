"""Benchmark of the draft step: NVFP4 64,064 x 2560 head GEMV + argmax, M = 1.

One step = one draft_head_top_tokens call (GEMV + argmax + dh_idx map) on a
fresh BF16 hidden state. Workload: V = 248,320, K = 2560, 64,026 kept ids
padded to 64,064 rows. L2 (129 MB) is defeated by rotating six copies of the
92.25 MB head (553.5 MB). The K timed steps are captured in one CUDA graph
(as a drafter replays its draft loop) and timed with CUDA events on the
launching stream; value = µs per draft step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only baseline here) on the same
workload: each step computes a bounded sample of the head's rows in fp64 and
is scaled to a full step.
With N > 1 (torchrun) every rank runs an independent replica (the draft head
does not shard on one box); value = max-over-ranks time / (N * K).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as syn  # noqa: E402

METRIC = "µs/draft step & HBM GB/s, NVFP4 64,064×2560 head GEMV+argmax, M=1"
WORKLOAD = "nvfp4 draft head 64,064x2560 (V=248,320, 64,026 kept), GEMV+argmax, M=1"
COPIES = 6
FALLBACK_HBM_GBS = 6800.0

# Algorithmic bytes of one draft step at M = 1: NVFP4 codes (64,064 x 1,280 B)
# + E4M3 block scales (64,064 x 160 B) + g (4 B) + h (2,560 x 2 B) + the id (4 B).
# The method needs dh_idx only for the winning row; the kernel stages all of it
# (256 KB, L2-resident from step to step) so that its argmax keys carry ids.
N_ROWS, K_HID = 64_064, 2_560
FLUSH_BYTES = 256 << 20                                   # 2 x the 129 MB L2
STEP_BYTES = N_ROWS * (K_HID // 2) + N_ROWS * (K_HID // 16) + 4 + 2 * K_HID + 4

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum, mean of two
# launches) of one launch of the M = 1 GEMV, from an ncu capture of
# `bench.py --profile`; reported only while the kernel sources still hash to
# kernel_sha (else null).
TRAFFIC = {"kernel_sha": "ce288d8c8815972c", "bytes_per_launch": 93_781_632}


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in ("dh_gemv_mma.cuh", "dh_epilogue.cuh", "dh_common.cuh", "dh_gemv_nvfp4p.cu", "dh_gemv_nvfp4p_ldg.cu"):
        with open(os.path.join(ROOT, "nvfp4_draft_head_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the GPU is under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows if len(r) >= 9
                          for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (all-reduce MAX over the default process
    group; x itself when there is no group)."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_step(ms_max: float, steps: int, world: int) -> float:
    """µs per draft step of the whole job: N replicas each ran `steps` steps in
    at most ms_max milliseconds, so N * steps steps took ms_max."""
    return ms_max * 1e3 / (steps * world)


def workload_host():
    c = syn.QWEN_64K
    W = syn.head_bf16(syn.SEED_HEAD_QWEN, c["V"], c["K"])
    keep = syn.keep_mask(syn.SEED_KEEP_64K, c["V"], c["n_kept"], c["forced"])
    return W, keep


def hidden_steps(n):
    return np.concatenate([syn.hidden_bf16(syn.hidden_seed(1, i), 1, K_HID) for i in range(n)])


def oracle_sample_steps(q, sf, g, hs, n_steps, sample_rows, budget_s=None):
    """Time the oracle's draft step on a bounded sample: step i computes the
    fp64 logits and argmax of `sample_rows` consecutive head rows (a rotating
    window); returns (seconds per full step, steps done)."""
    import oracle
    n_win = N_ROWS // sample_rows
    t_total, done = 0.0, 0
    for i in range(n_steps):
        w = i % n_win
        r0 = w * sample_rows
        h = hs[i % hs.shape[0]][None]
        t0 = time.perf_counter()
        y, _ = oracle.gemv(oracle.FMT_NVFP4, q[r0:r0 + sample_rows], sf[r0:r0 + sample_rows], g, h,
                           want_abs=False)
        oracle.top_tokens(y, None)
        t_total += time.perf_counter() - t0
        done += 1
        if budget_s is not None and t_total >= budget_s:
            break
    return t_total / done * (N_ROWS / sample_rows), done


def oracle_all_cores(q, sf, g, hs, budget_s=10.0):
    """The oracle's full draft step (fp64 GEMV over all rows + argmax) with the
    rows split evenly over one Python thread per host core (the oracle is C
    behind ctypes, which releases the GIL). Returns (seconds per step, steps,
    threads)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    n_thr = max(1, os.cpu_count() or 1)
    bounds = [(N_ROWS * i // n_thr, N_ROWS * (i + 1) // n_thr) for i in range(n_thr)]

    def part(args):
        (r0, r1), h = args
        y, _ = oracle.gemv(oracle.FMT_NVFP4, q[r0:r1], sf[r0:r1], g, h, want_abs=False)
        return r0, y[0]

    t_total, done = 0.0, 0
    with ThreadPoolExecutor(n_thr) as ex:
        while t_total < budget_s:
            h = hs[done % hs.shape[0]][None]
            t0 = time.perf_counter()
            y = np.empty(N_ROWS)
            for r0, yr in ex.map(part, [(b, h) for b in bounds]):
                y[r0:r0 + yr.size] = yr
            oracle.top_tokens(y[None], None)
            t_total += time.perf_counter() - t0
            done += 1
    return t_total / done, done, n_thr


def bench_config(world: int) -> dict:
    """The workload description both arms print."""
    return {"workload": WORKLOAD, "M": 1, "V": 248_320, "K": K_HID, "N": N_ROWS, "n_kept": 64_026,
            "head_copies": COPIES, "l2": "inputs larger than L2: 6 rotating head copies (553.5 MB > 4 x 129 MB)",
            "timing": "one CUDA graph of K steps, CUDA events",
            "parallelism": "replicas" if world > 1 else "single"}


def emit(obj):
    print(json.dumps(obj), flush=True)


def run_reference(args, world, rank):
    """The CPU oracle on this host's cores, same workload, metric and unit."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    W, keep = workload_host()
    idx, nk = oracle.build_index(keep)
    q, sf, g = oracle.nvfp4_quantize(W, idx)
    hs = hidden_steps(min(64, args.warmup + args.steps))
    sample = N_ROWS // 16
    oracle_sample_steps(q, sf, g, hs, args.warmup, sample)
    sec, done = oracle_sample_steps(q, sf, g, hs, args.steps, sample)
    us = sec * 1e6
    cpu = {"value": us, "unit": "us/step", "cores": 1, "kind": "oracle",
           "sample": f"each step: fp64 GEMV+argmax over {sample} of {N_ROWS} rows (rotating window), "
                     f"scaled x{N_ROWS // sample}"}
    emit({"impl": "reference", "metric": METRIC, "value": us, "unit": "us/step", "n_gpus": world,
          "steps": done, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
          "config": bench_config(world),
          "cpu_baseline": cpu,
          "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})


def run_ours(args, world, rank, local):
    import torch

    import nvfp4_draft_head_gb300 as dh
    from nvfp4_draft_head_gb300 import build

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
    build.build()
    lib_loaded = dh.lib()

    W, keep = workload_host()
    Wd = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    head = dh.nvfp4_head(Wd, keep)
    del Wd
    heads = [head] + [head.with_storage(head.q.clone()) for _ in range(COPIES - 1)]
    K, Wm = args.steps, args.warmup
    hs_host = hidden_steps(Wm + K)
    hs = torch.from_numpy(hs_host.view(np.int16)).to(dev).view(torch.bfloat16)
    ids = torch.empty((Wm + K, 1), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    check_leg = rank == 0 and world == 1 and not args.profile
    if not check_leg:
        del W                                             # the oracle leg below needs it

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    if args.profile:
        # Short run for a profiler: W + K eager steps over the rotating copies,
        # nothing else (no graph, no clock sampling, no end-to-end leg).
        with torch.cuda.stream(s):
            for i in range(Wm + K):
                heads[i % COPIES].top_tokens(hs[i:i + 1], ids=ids[i])
        s.synchronize()
        assert head.device_error() == 0
        if rank == 0:
            emit({"profile_run": True, "steps": K, "warmup": Wm})
        return
    with torch.cuda.stream(s):
        for i in range(Wm):                               # untimed warm-up steps
            heads[i % COPIES].top_tokens(hs[i:i + 1], ids=ids[i])
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for i in range(Wm, Wm + K):
                heads[i % COPIES].top_tokens(hs[i:i + 1], ids=ids[i])
        graph.replay()                                    # untimed: uploads the graph
    s.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.perf_counter() + 1.5                     # sustained load around the timed region
    with torch.cuda.stream(s):
        while time.perf_counter() < t_end:
            graph.replay()
            s.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        graph.replay()
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        for _ in range(3):                                # keep load on while the sampler catches up
            graph.replay()
        s.synchronize()
    clocks = sampler.stop()
    if world > 1:
        ms = max_over_ranks(ms, dev)
        torch.distributed.barrier()
    assert head.device_error() == 0

    # L2-flush cross-check: one head copy; before each step a 256 MB write
    # (2 x L2) evicts the head from L2, and the step alone is timed with events
    # around it. The flush sits between consecutive steps, so this leg has no
    # overlap between steps (each one starts cold and ends before the next).
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    n_fl = min(K, 200)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_fl)]
    with torch.cuda.stream(s):
        for i in range(n_fl):
            flush.fill_(i & 0xFF)
            evs[i][0].record(s)
            head.top_tokens(hs[Wm + i:Wm + i + 1], ids=ids[Wm + i])
            evs[i][1].record(s)
        s.synchronize()
    fl_us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    l2_flush = {"median_us_per_step": fl_us[len(fl_us) // 2], "mean_us_per_step": sum(fl_us) / len(fl_us),
                "steps": n_fl, "flush_bytes": FLUSH_BYTES,
                "how": "one head copy; a 256 MB write before each step; each step timed alone with CUDA events"}
    del flush

    # End to end through the public call with host buffers
    # (draft_head_top_tokens_host): per step, one call copies the hidden state
    # from pinned host memory, runs the draft step and copies the id back.
    h_pin = torch.from_numpy(hs_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_pin = torch.empty((Wm + K, 1), dtype=torch.int32).pin_memory()
    with torch.cuda.stream(s):
        for i in range(Wm):
            heads[i % COPIES].top_tokens_host(h_pin[i:i + 1], ids_pin[i])
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(s)
        for i in range(Wm, Wm + K):
            heads[i % COPIES].top_tokens_host(h_pin[i:i + 1], ids_pin[i])
        f1.record(s)
        torch.cuda.synchronize()
        ms_e2e = f0.elapsed_time(f1)
    if world > 1:
        ms_e2e = max_over_ranks(ms_e2e, dev)
    e2e_ok = bool(np.array_equal(ids_pin[Wm:].numpy(), ids[Wm:].cpu().numpy()))

    # CPU-oracle leg (rank 0, one GPU): the oracle quantises the same head, the
    # GPU's packed head must equal it byte for byte and the first timed graph
    # steps' ids must meet the tolerance rule; then the oracle's own draft step
    # is timed on this host's cores.
    cpu = cpu_all = parity = None
    if check_leg:
        import oracle
        oracle.build()
        idx_o, nk = oracle.build_index(keep)
        q_o, sf_o, g_o = oracle.nvfp4_quantize(W, idx_o)
        del W
        N_, Kh = q_o.shape
        nwin = 2 * Kh // 128
        packed_o = np.concatenate(
            [q_o.reshape(N_ // 16, 16, nwin, 64).transpose(0, 2, 1, 3).reshape(N_ // 16, nwin, 1024),
             sf_o.reshape(N_ // 16, 2, 8, nwin, 4, 2).transpose(0, 3, 2, 4, 1, 5).reshape(N_ // 16, nwin, 128)],
            axis=2)
        exact = (np.array_equal(head.q.cpu().numpy(), packed_o) and head.scale.cpu().numpy()[0] == g_o)
        n_chk = min(3, K)
        got = ids[Wm:Wm + n_chk, 0].cpu().numpy()
        ok = True
        for i in range(n_chk):
            y, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, hs_host[Wm + i:Wm + i + 1])
            r = int(np.argmax(y[0, :nk]))
            j = int(np.nonzero(idx_o[:nk] == got[i])[0][0]) if got[i] in idx_o[:nk] else -1
            t = lambda n: 2e-3 * A[0, n] + 1e-5
            ok &= (j == r) or (j >= 0 and y[0, r] - y[0, j] <= t(r) + t(j))
        parity = {"quantize_bit_exact": bool(exact), "timed_steps_checked": n_chk, "ids_within_tolerance": bool(ok)}
        if not (exact and ok):
            emit({"error": "parity failed", "parity": parity})
            sys.exit(1)
        sec, done = oracle_sample_steps(q_o, sf_o, g_o, hs_host, 10_000, N_ROWS // 16, budget_s=12.0)
        cpu = {"value": sec * 1e6, "unit": "us/step", "cores": 1, "kind": "oracle",
               "sample": f"{done} steps, each an fp64 GEMV+argmax over {N_ROWS // 16} of {N_ROWS} rows "
                         f"(rotating window) scaled x16; single-threaded C"}
        sec_a, done_a, thr = oracle_all_cores(q_o, sf_o, g_o, hs_host, budget_s=10.0)
        cpu_all = {"value": sec_a * 1e6, "unit": "us/step", "cores": thr, "kind": "oracle",
                   "sample": f"{done_a} full steps (all {N_ROWS} rows, fp64 GEMV + argmax), rows split over "
                             f"{thr} threads"}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    us_step = ms * 1e3 / K
    value = whole_job_us_per_step(ms, K, world)
    gbs = STEP_BYTES / (us_step * 1e-6) / 1e9
    peak, peak_src = hbm_peak()
    sha = kernel_sha()
    traffic = TRAFFIC["bytes_per_launch"] if TRAFFIC["kernel_sha"] == sha else None
    emit({"metric": METRIC, "value": value, "unit": "us/step", "n_gpus": world, "steps": K, "warmup": Wm,
          "ms_per_step": us_step / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
          "dtype": "f32", "data": "synthetic",
          "config": bench_config(world),
          "hbm_gbs": gbs,
          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "peak_source": peak_src,
                       "unit": "GB/s", "frac": gbs / peak, "traffic": traffic,
                       "kernel": "gemv_mma_kernel<NVFP4 packed, K=2560, M=1> (top tokens)",
                       "bytes_per_launch": STEP_BYTES},
          "cpu_baseline": cpu, "cpu_baseline_all_cores": cpu_all,
          "e2e": {"value": whole_job_us_per_step(ms_e2e, K, world), "unit": "us/step", "h2d_bytes_per_step": 2 * K_HID,
                  "d2h_bytes_per_step": 4, "ids_match_graph": e2e_ok, "call": "draft_head_top_tokens_host"},
          "l2_flush_leg": l2_flush,
          "gpu_launches": K, "clocks": clocks, "parity": parity,
          "library": os.path.relpath(dh.library_path(), ROOT), "kernel_sha": sha})
    if world > 1:
        torch.distributed.destroy_process_group()
    del lib_loaded


def run_profile_case(args):
    """Eager draft steps of one secondary workload for a profiler (no timing,
    no output but one line): the batch sweep on the NVFP4 head (--drafts M),
    the 98,304-row FP8 head (W8A16 or W8A8), or the fc-sized NVFP4 linear."""
    import torch

    import nvfp4_draft_head_gb300 as dh
    from nvfp4_draft_head_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M = args.drafts
    hs = torch.from_numpy(np.concatenate([syn.hidden_bf16(7000 + i, 16, K_HID) for i in range(8)]).view(np.int16)
                          ).to(dev).view(torch.bfloat16).reshape(8, 16, K_HID)
    W, keep = workload_host()
    Wd = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    del W
    if args.profile_case == "nvfp4":
        h0 = dh.nvfp4_head(Wd, keep)
        units = [h0] + [h0.with_storage(h0.q.clone()) for _ in range(COPIES - 1)]
    elif args.profile_case in ("fp8", "w8a8"):
        c = syn.FP8_98K
        k8 = syn.keep_mask(syn.SEED_KEEP_98K, c["V"], c["n_kept"], c["forced"])
        h8 = dh.fp8_head(Wd, k8, w8a8=args.profile_case == "w8a8")
        units = [h8] + [h8.with_storage(h8.q.clone()) for _ in range(2)]
    else:  # linear: fc 5,120 -> 2,560, 70 copies (520 MB)
        Wl = torch.from_numpy(syn.head_bf16(4000 + 5120, 2560, 5120).view(np.int16)).to(dev).view(torch.bfloat16)
        l0 = dh.NVFP4Linear(Wl)
        units = [l0] + [l0.with_storage(l0.packed.clone()) for _ in range(69)]
        hs = torch.from_numpy(np.concatenate([syn.hidden_bf16(7200 + i, 16, 5120) for i in range(8)]).view(np.int16)
                              ).to(dev).view(torch.bfloat16).reshape(8, 16, 5120)
    del Wd
    ids = torch.empty(M, dtype=torch.int32, device=dev)
    for i in range(args.warmup + args.steps):
        u = units[i % len(units)]
        if args.profile_case == "linear":
            u(hs[i % 8, :M])
        else:
            u.top_tokens(hs[i % 8, :M], ids=ids)
    torch.cuda.synchronize()
    assert units[0].device_error() == 0
    emit({"profile_run": True, "case": args.profile_case, "drafts": M, "steps": args.steps, "warmup": args.warmup})


def run_suite(args):
    """Secondary measurements (one JSON line each) of the other workloads:
    the FP8 98,304-row head, the batch sweep, the BF16 full-vocabulary head,
    the head build, and the tiny head. Same timing method as the main line
    (one CUDA graph of `steps` calls, inputs rotated over copies > 4 x L2)."""
    import torch

    import nvfp4_draft_head_gb300 as dh
    from nvfp4_draft_head_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    steps = max(50, min(args.steps, 500))

    def graph_us(calls):
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for c in calls[:3]:
                c()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for c in calls:
                    c()
            g.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            s.synchronize()
        return e0.elapsed_time(e1) * 1e3 / len(calls)

    def line(name, us, nbytes, extra=None):
        d = {"suite": name, "us_per_call": us, "gbs": nbytes / (us * 1e-6) / 1e9, "bytes_per_call": nbytes}
        if extra:
            d.update(extra)
        emit(d)

    W, keep = workload_host()
    Wd = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    hs = torch.from_numpy(hidden_steps(64).view(np.int16)).to(dev).view(torch.bfloat16)
    hsM = torch.from_numpy(np.concatenate([syn.hidden_bf16(7000 + i, 16, K_HID) for i in range(8)]).view(np.int16)
                           ).to(dev).view(torch.bfloat16).reshape(8, 16, K_HID)

    # head build (quantise + pack), timed as single calls after a warm-up
    idx_np, nk = dh.draft_head_build_index(keep)
    idx = torch.from_numpy(idx_np).to(dev)
    q = torch.empty((N_ROWS, K_HID // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty((N_ROWS, K_HID // 16), dtype=torch.uint8, device=dev)
    gsc = torch.empty(1, dtype=torch.float32, device=dev)
    packed = torch.empty((N_ROWS // 16, K_HID // 128, 1152), dtype=torch.uint8, device=dev)
    nb = dh.lib().draft_head_quantize_workspace_bytes()
    ws = dh._workspace(nb, dev)
    st = torch.cuda.current_stream().cuda_stream

    def quant():
        dh.lib().nvfp4_quantize_rows(Wd.data_ptr(), Wd.shape[0], K_HID, idx.data_ptr(), N_ROWS, q.data_ptr(),
                                     sf.data_ptr(), gsc.data_ptr(), ws.data_ptr(), nb,
                                     torch.cuda.current_stream().cuda_stream)

    def pack():
        dh.lib().nvfp4_pack_head(q.data_ptr(), sf.data_ptr(), N_ROWS, K_HID, packed.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    del st
    for _ in range(3):
        quant()
        pack()
    torch.cuda.synchronize()
    qbytes = 2 * (N_ROWS * K_HID * 2 + N_ROWS * 4) + N_ROWS * (K_HID // 2 + K_HID // 16) + 4
    line("nvfp4 gather+quantise 64,064 x 2560", graph_us([quant] * 20), qbytes)
    line("nvfp4 repack 64,064 x 2560", graph_us([pack] * 20), 2 * N_ROWS * (K_HID // 2 + K_HID // 16))

    # batch sweep on the packed head (six rotating copies)
    head = dh.nvfp4_head(Wd, keep)
    heads = [head] + [head.with_storage(head.q.clone()) for _ in range(COPIES - 1)]
    hb = N_ROWS * (K_HID // 2 + K_HID // 16) + 4
    for M in (1, 2, 4, 8, 16):
        ids = torch.empty(M, dtype=torch.int32, device=dev)
        out = torch.empty((M, 248_320), dtype=torch.float32, device=dev)
        calls = [(lambda i=i: heads[i % COPIES].top_tokens(hsM[i % 8, :M], ids=ids)) for i in range(steps)]
        line(f"nvfp4 top_tokens M={M}", graph_us(calls), hb + M * (2 * K_HID + 4), {"M": M})
        calls = [(lambda i=i: heads[i % COPIES].compute_logits(hsM[i % 8, :M], out=out)) for i in range(steps)]
        line(f"nvfp4 compute_logits M={M}", graph_us(calls), hb + M * (2 * K_HID + 4 * 248_320), {"M": M})
    del heads, head

    # FP8 98,304-row head (three rotating copies = 755 MB)
    c = syn.FP8_98K
    keep8 = syn.keep_mask(syn.SEED_KEEP_98K, c["V"], c["n_kept"], c["forced"])
    h8 = dh.fp8_head(Wd, keep8)
    h8s = [h8] + [h8.with_storage(h8.q.clone()) for _ in range(2)]
    fb = h8.N * K_HID + 4
    for M in (1, 4):
        ids = torch.empty(M, dtype=torch.int32, device=dev)
        out = torch.empty((M, 248_320), dtype=torch.float32, device=dev)
        calls = [(lambda i=i: h8s[i % 3].top_tokens(hsM[i % 8, :M], ids=ids)) for i in range(steps)]
        line(f"fp8 98,304 top_tokens M={M}", graph_us(calls), fb + M * (2 * K_HID + 4), {"M": M})
        calls = [(lambda i=i: h8s[i % 3].compute_logits(hsM[i % 8, :M], out=out)) for i in range(steps)]
        line(f"fp8 98,304 compute_logits M={M}", graph_us(calls), fb + M * (2 * K_HID + 4 * 248_320), {"M": M})
    # the same head run W8A8 (per-token FP8 hidden states quantised inside the step)
    w8 = [dh.DraftHead(dh.DH_FMT_FP8_W8A8, x.V, x.q, x.idx, x.n_kept, scale=x.scale, idx_ascending=True)
          for x in h8s]
    for M in (1, 4, 16):
        ids = torch.empty(M, dtype=torch.int32, device=dev)
        out = torch.empty((M, 248_320), dtype=torch.float32, device=dev)
        calls = [(lambda i=i: w8[i % 3].top_tokens(hsM[i % 8, :M], ids=ids)) for i in range(steps)]
        line(f"fp8 w8a8 98,304 top_tokens M={M}", graph_us(calls), fb + M * (2 * K_HID + 4), {"M": M})
        calls = [(lambda i=i: w8[i % 3].compute_logits(hsM[i % 8, :M], out=out)) for i in range(steps)]
        line(f"fp8 w8a8 98,304 compute_logits M={M}", graph_us(calls), fb + M * (2 * K_HID + 4 * 248_320),
             {"M": M})
    del h8s, h8, w8

    # BF16 full-vocabulary head, the stock drafter read (1.27 GB > L2)
    hf = dh.bf16_full_head(Wd)
    ids = torch.empty(1, dtype=torch.int32, device=dev)
    calls = [(lambda i=i: hf.top_tokens(hs[i % 64: i % 64 + 1], ids=ids)) for i in range(min(steps, 200))]
    line("bf16 248,320 x 2560 top_tokens M=1", graph_us(calls), 248_320 * K_HID * 2 + 2 * K_HID + 4)
    # truncated 40,960-row BF16 draft head read in place (six copies = 1.26 GB > L2)
    tr = [dh.bf16_truncated_head(Wd[i * 40_960:], 40_960) for i in range(6)]
    for M in (1, 4):
        ids = torch.empty(M, dtype=torch.int32, device=dev)
        calls = [(lambda i=i: tr[i % 6].top_tokens(hsM[i % 8, :M], ids=ids)) for i in range(steps)]
        line(f"bf16 truncated 40,960 x 2560 top_tokens M={M}", graph_us(calls), 40_960 * K_HID * 2 + M * (2 * K_HID + 4),
             {"M": M})

    # NVFP4 W4A16 MTP-block linears (synthetic shapes around a 2,560-wide block),
    # each rotated over copies totalling > 4 x L2
    for K_in, N_out, name in ((5120, 2560, "fc"), (2560, 4608, "qkv"), (4096, 2560, "o_proj"),
                              (2560, 1024, "shared-expert gate/up"), (512, 2560, "shared-expert down")):
        Wl = torch.from_numpy(syn.head_bf16(4000 + K_in, N_out, K_in).view(np.int16)).to(dev).view(torch.bfloat16)
        l0 = dh.NVFP4Linear(Wl)
        nb = N_out * (K_in // 2 + K_in // 16)
        lins = [l0] + [l0.with_storage(l0.packed.clone()) for _ in range(max(1, (600 << 20) // nb) - 1)]
        xs = torch.from_numpy(np.concatenate([syn.hidden_bf16(7200 + i, 16, K_in) for i in range(8)]).view(np.int16)
                              ).to(dev).view(torch.bfloat16).reshape(8, 16, K_in)
        for M in (1, 16):
            y = torch.empty((M, N_out), dtype=torch.float32, device=dev)
            calls = [(lambda i=i: lins[i % len(lins)](xs[i % 8, :M], y=y)) for i in range(steps)]
            line(f"nvfp4 linear {name} {K_in}->{N_out} M={M}", graph_us(calls), nb + 4 + M * (2 * K_in + 4 * N_out),
                 {"M": M, "copies": len(lins)})
        del lins, l0, Wl

    # tiny head (L2-resident, latency-bound)
    ct = syn.TINY
    Wt = torch.from_numpy(syn.head_bf16(syn.SEED_HEAD_TINY, ct["V"], ct["K"]).view(np.int16)).to(dev).view(torch.bfloat16)
    ht = dh.nvfp4_head(Wt, syn.keep_mask(syn.SEED_KEEP_TINY, ct["V"], ct["n_kept"], ct["forced"]))
    htid = torch.from_numpy(syn.hidden_bf16(1, 64, ct["K"]).view(np.int16)).to(dev).view(torch.bfloat16)
    calls = [(lambda i=i: ht.top_tokens(htid[i % 64: i % 64 + 1], ids=ids)) for i in range(steps)]
    line("tiny nvfp4 4,032 x 256 top_tokens M=1", graph_us(calls), ht.N * (ct["K"] // 2 + ct["K"] // 16))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--profile", action="store_true",
                    help="eager steps only, for ncu (prints no measurement)")
    ap.add_argument("--profile-case", choices=("nvfp4", "fp8", "w8a8", "linear"), default=None,
                    help="with --profile: a secondary workload (NVFP4 head at --drafts M, the 98,304-row FP8 "
                         "head W8A16 / W8A8, or the fc-sized NVFP4 linear)")
    ap.add_argument("--drafts", type=int, default=1, help="drafts per step for --profile-case")
    ap.add_argument("--suite", action="store_true",
                    help="one line per secondary workload (FP8 head, batch sweep, BF16 head, head build, tiny)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.profile and args.profile_case:
        run_profile_case(args)
        return
    if args.suite:
        run_suite(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
