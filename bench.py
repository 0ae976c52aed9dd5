"""Benchmark: paged GQA decode KV GB/s, % of HBM peak and tokens/s per layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one decode call (block-table walk, TMA page staging, q K^T, online
softmax, P V, split-KV merge) over one batch of the workload, with every input
resident in HBM.  The default workload is the Llama-3-8B layer shape: B=64
sequences, lengths uniform in [128, 4096], Hq=32, Hkv=8, D=128, 16-token
blocks, bf16, a pool of ceil(1.1 * used) blocks with a seeded shuffled block
table.  Its K/V (about 0.6 GB) is larger than L2, so no flush is needed between
steps.  The K timed steps are captured as one CUDA graph and replayed, as a
serving loop replays its decode step (--launch stream launches them one by one
from Python instead).  Rank 0 prints one JSON line.

--impl reference times the float64 CPU oracle on the host cores instead (the
comparison arm), over the same workload.
Multi-GPU: every rank runs its own replica of the workload (seed + rank), no
data-path collective; value = all ranks' bytes / max time.  `--gpus N` with
N > 1 outside a launcher re-launches this script under torch.distributed.run
with N processes on this node (127.0.0.1); under a launcher the world size
must equal N.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gen  # noqa: E402
from paged_gqa_decode_04_gb300 import accounting  # noqa: E402

METRIC = "paged GQA decode KV GB/s and % of GB300 HBM peak; tokens/s per layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "paged_gqa_decode_04_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def describe(w):
    spec = gen.CONFIGS[w.name]
    return ("%s: B=%d, Hq=%d, Hkv=%d (G=%d), D=%d, block_size=%d, %s, lengths %s, "
            "pool %d blocks, seed %d" % (w.name, w.B, w.Hq, w.Hkv, w.G, w.D, w.block_size,
                                         w.dtype, spec["lens"] if not isinstance(spec["lens"], list)
                                         else "fixed", w.num_blocks, w.seed))


def workload_bytes(w, q_len=1, window=0):
    """Algorithmic bytes of one step over workload w (8-bit pages with a scale
    per block and KV head also read those scales)."""
    elt, q_elt = accounting.ELT[w.dtype], accounting.Q_ELT[w.dtype]
    pb = w.k_scale is not None and w.k_scale.dim() == 2
    if q_len == 1 and window == 0:
        return accounting.algorithmic_bytes(w.lens_np, w.Hq, w.Hkv, w.D, w.block_size, elt, q_elt,
                                            block_scales=pb)
    return accounting.algorithmic_bytes_ex(w.lens_np, w.Hq, w.Hkv, w.D, w.block_size, elt, q_len,
                                           window, q_elt, block_scales=pb)


def oracle_q8(oracle, w, q, k, v, table, lens):
    """The oracle on 8-bit pages of w (e4m3 or int8 codes, either scale form)."""
    return oracle.decode_q8_f64(q, k, v, "e4m3" if w.dtype == "fp8" else "int8",
                                w.k_scale.cpu().numpy(), w.v_scale.cpu().numpy(), table, lens,
                                w.scale)


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


_COMMENT_OR_STRING = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"', re.S)


def kernel_hash(csrc=CSRC):
    """Hash of the decode kernel's code: every device-side source of it
    (decode_tma*, partition.cuh, pgd_internal.h) with comments dropped and
    whitespace collapsed, so that an edit of comments alone keeps it."""
    names = sorted(n for n in os.listdir(csrc)
                   if (n.startswith("decode_tma") and n.endswith((".cu", ".cuh")))
                   or n in ("partition.cuh", "pgd_internal.h"))
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(csrc, n)) as f:
            text = f.read()
        code = _COMMENT_OR_STRING.sub(lambda m: m.group(0) if m.group(0)[0] == '"' else " ", text)
        h.update(n.encode() + b"\0" + " ".join(code.split()).encode() + b"\0")
    return h.hexdigest()[:16]


def ncu_traffic(config):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source and this workload; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            doc = json.load(f)
        ent = doc.get(config)
        if ent and ent.get("kernel_sha") == kernel_hash():
            return int(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples while it runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w", prefix="bench_clocks_", suffix=".csv",
                                                 delete=False)
            self.path = self.f.name
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index),
                                          "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        try:
            with open(self.path) as f:
                lines = f.readlines()
            os.unlink(self.path)
        except OSError:
            return None
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r[2] > 1.5 * min(x[2] for x in rows)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[3][1:5])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(busy)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def free_port():
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def relaunch_cmd(argv, gpus, port):
    """This script under torch.distributed.run: `gpus` ranks on this node."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            "--nproc-per-node", str(gpus), "--master-addr", "127.0.0.1",
            "--master-port", str(port), os.path.abspath(__file__)] + list(argv)


def gather_over_ranks(x, world, device):
    """Every rank's value of x, in rank order (on every rank)."""
    if world == 1:
        return [x]
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    parts = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(parts, t)
    return [float(p.item()) for p in parts]


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(config, rank):
    """Each rank runs its own replica of the workload, drawn with seed + rank."""
    return gen.CONFIGS[config]["seed"] + rank


def whole_job_gbs(nbytes, t_ms, world):
    """Bytes all ranks moved (each its own replica) over the slowest rank's time."""
    return world * nbytes / (t_ms * 1e-3) / 1e9


def cold_median_ms(step, stream, dev, reps=50):
    """Median device time of `reps` single launches of `step`, each preceded by
    a read of a buffer twice the L2 size, so that the launch finds none of its
    inputs in L2 (a read rather than a write: a written buffer would leave L2
    full of dirty lines whose write-back the timed launch would pay for);
    events bracket the launch alone."""
    if reps <= 0:
        return None
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (126 << 20)
    flush = torch.ones(2 * l2 // 4, dtype=torch.int32, device=dev)
    acc = torch.zeros((), dtype=torch.int64, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            acc += flush.sum()
            e0.record(stream)
            step()
            e1.record(stream)
    torch.cuda.synchronize()
    if int(acc.item()) != reps * flush.numel():
        raise RuntimeError("L2 flush read back a wrong sum")
    times = [e0.elapsed_time(e1) for e0, e1 in evs]
    del flush
    return statistics.median(times)


def launch_note(args):
    if args.launch == "graph":
        return "the %d timed steps captured as one CUDA graph, replayed once" % args.steps
    return "the %d timed steps launched one by one on one stream" % args.steps


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_oracle_rate(w, budget_s, threads=0):
    """Run the oracle over the whole workload until `budget_s` has passed, on
    `threads` host cores (0: all); returns (GB/s over algorithmic bytes,
    sample, cores, sequences/s)."""
    import oracle

    oracle.set_num_threads(threads if threads > 0 else host_cores())

    q, k, v = gen.to_numpy_bits(w.q), gen.to_numpy_bits(w.k_pool), gen.to_numpy_bits(w.v_pool)
    elt, q_elt = accounting.ELT[w.dtype], accounting.Q_ELT[w.dtype]
    nbytes = workload_bytes(w)
    if w.dtype in gen.Q8:
        run = lambda: oracle_q8(oracle, w, q, k, v, w.table_np, w.lens_np)
    else:
        run = lambda: oracle.decode_f64(q, k, v, w.table_np, w.lens_np, w.scale)
    reps = 0
    t0 = time.perf_counter()
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    sample = ("%d full pass(es) of the workload (all %d x %d rows) in %.1f s on %d host core(s)"
              % (reps, w.B, w.Hq, dt, oracle.num_threads()))
    return nbytes * reps / dt / 1e9, sample, oracle.num_threads(), w.B * reps / dt


def run_reference(args, world, rank):
    """The comparison arm: the float64 CPU oracle as it stands."""
    if rank != 0:
        return
    w = gen.make(args.config, device="cpu")
    elt, q_elt = accounting.ELT[w.dtype], accounting.Q_ELT[w.dtype]
    nbytes = workload_bytes(w)
    import oracle

    oracle.set_num_threads(args.cpu_threads if args.cpu_threads > 0 else host_cores())
    cores = oracle.num_threads()
    q, k, v = gen.to_numpy_bits(w.q), gen.to_numpy_bits(w.k_pool), gen.to_numpy_bits(w.v_pool)
    # One step = the oracle over a bounded sample: every sequence, a subset of
    # query heads (whole KV groups) so that K+W steps fit in a few minutes.
    if w.dtype in gen.Q8:
        # 8-bit pages: every query head of the first B/8 sequences per step
        nb = max(1, w.B // 8)
        step = lambda: oracle_q8(oracle, w, q[:nb], k, v, w.table_np[:nb], w.lens_np[:nb])
        frac = accounting.algorithmic_bytes(w.lens_np[:nb], w.Hq, w.Hkv, w.D, w.block_size, elt,
                                            q_elt) / accounting.algorithmic_bytes(
            w.lens_np, w.Hq, w.Hkv, w.D, w.block_size, elt, q_elt)
        sample = ("each step: sequences 0..%d of %d, every query head, float64, %d host "
                  "core(s)" % (nb - 1, w.B, cores))
    else:
        heads = max(w.G, min(w.Hq, (w.Hq // 8) // w.G * w.G or w.G))
        rows = np.array([[b, h] for b in range(w.B) for h in range(heads)], dtype=np.int32)
        frac = heads / w.Hq
        step = lambda: oracle.decode_rows_f64(q, k, v, w.table_np, w.lens_np, w.scale, rows)
        sample = ("each step: every sequence, query heads 0..%d of %d (%.1f%% of the rows), "
                  "float64, %d host core(s)" % (heads - 1, w.Hq, 100 * frac, cores))
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes * frac / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w), "parallelism": "%d host core(s)" % cores},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import paged_gqa_decode_04_gb300 as pgd

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = gen.make(args.config, device=dev, seed=replica_seed(args.config, rank))
    elt, q_elt = accounting.ELT[w.dtype], accounting.Q_ELT[w.dtype]
    nbytes = workload_bytes(w)
    pool = pgd.PagedKVPool(w.k_pool, w.v_pool, w.k_scale, w.v_scale)
    out = torch.empty_like(w.q)
    ws = pgd.alloc_workspace(pool, w.B, w.Hq, 0)
    stream = torch.cuda.current_stream(dev)

    def step(s=None):
        pgd.paged_gqa_decode(pool, w.q, w.block_table, w.seq_lens, w.scale, out=out,
                             workspace=ws, stream=s or stream)

    op_note = "decode: one query token per sequence"
    if args.op == "decode_ex":
        # q_len query tokens per sequence (the last q_len cached ones), optional window
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed + 7)
        q_ex = torch.randn((w.B, args.q_len, w.Hq, w.D), generator=g, device=dev).to(w.q.dtype)
        out = torch.empty_like(q_ex)
        nbytes = workload_bytes(w, args.q_len, args.window)
        ws = torch.zeros(max(256, pgd.paged_gqa_workspace_size_ex(pool, w.B, args.q_len, w.Hq)),
                         dtype=torch.uint8, device=dev)

        def step(s=None):
            pgd.paged_gqa_decode_ex(pool, q_ex, w.block_table, w.seq_lens, w.scale,
                                    window=args.window, out=out, workspace=ws, stream=s or stream)

        op_note = "decode_ex: %d query tokens per sequence, window %d" % (args.q_len, args.window)
    elif args.op == "append":
        # store one new token per sequence (K and V rows) at distinct slots
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed + 9)
        k_new = torch.randn((w.B, w.Hkv, w.D), generator=g, device=dev).to(w.k_pool.dtype)
        v_new = torch.randn((w.B, w.Hkv, w.D), generator=g, device=dev).to(w.k_pool.dtype)
        slots = torch.arange(w.B, dtype=torch.int32, device=dev) * w.block_size
        nbytes = 2 * 2 * k_new.numel() * k_new.element_size() + 4 * w.B

        def step(s=None):
            pgd.paged_kv_append(pool, k_new, v_new, slots, stream=s or stream)

        op_note = "append: one new token per sequence (read + write of K and V rows)"

    # kernels one step launches: the decode, plus the run merge when the plan
    # merges split runs in a second kernel (or the float32 path's merge kernel)
    merge = "fused"
    kernels_per_step = 1
    if args.op != "append":
        plan = pgd.paged_gqa_plan(w.k_pool.dtype, w.Hkv, w.D, w.B, w.Hq,
                                  q_len=args.q_len if args.op == "decode_ex" else 1,
                                  window=args.window if args.op == "decode_ex" else 0)
        merge = plan["merge"]
        kernels_per_step = 2 if merge in ("separate", "merge kernel") else 1

    step()
    status = pgd.paged_gqa_get_error(pool, stream)
    if status != 0:
        raise RuntimeError("device error: %s" % pgd.strerror(status))

    if args.profile:
        # exactly W + K launches of the step and nothing else, for profilers
        for _ in range(args.warmup + args.steps):
            step()
        torch.cuda.synchronize()
        status = pgd.paged_gqa_get_error(pool, stream)
        if rank == 0:
            print(json.dumps({"profile_run": args.config, "launch_steps": args.warmup + args.steps,
                              "status": pgd.strerror(status)}), flush=True)
        if status != 0:
            raise RuntimeError("device error: %s" % pgd.strerror(status))
        return

    # warm-up: at least W steps and at least 0.5 s, so the clock sampler sees load
    with ClockSampler(local) as clk:
        t_warm = time.perf_counter()
        n = 0
        while n < args.warmup or time.perf_counter() - t_warm < 0.5:
            step()
            n += 1
            if n % 64 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        graph = None
        if args.launch == "graph":
            # the K timed steps as one CUDA graph (as a serving loop replays its
            # decode step); replayed once untimed first
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(graph, stream=cap):
                    for _ in range(args.steps):
                        step(cap)
            stream.wait_stream(cap)
            graph.replay()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for _ in range(args.steps):
                step()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
    t_ms = ev0.elapsed_time(ev1) / args.steps
    rank_ms = gather_over_ranks(t_ms, world, dev)
    t_ms = max(rank_ms)
    status = pgd.paged_gqa_get_error(pool, stream)
    if status != 0:
        raise RuntimeError("device error: %s" % pgd.strerror(status))
    # L2-cold figure: single launches, each after a read of twice the L2 size
    # on the same stream, events around the launch alone; median over 50
    cold_ms = cold_median_ms(step, stream, dev, reps=args.cold_reps)
    cold_ms = max_over_ranks(cold_ms, world, dev) if cold_ms is not None else None

    if args.op != "decode":
        if rank == 0:
            peak, peak_src = peak_hbm()
            gbs = whole_job_gbs(nbytes, t_ms, world)
            print(json.dumps({
                "metric": METRIC, "op": args.op, "value": round(gbs, 2), "unit": "GB/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(t_ms, 5), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
                "config": {"workload": describe(w), "op": op_note,
                           "launch": launch_note(args), "algorithmic_bytes_per_step": nbytes,
                           "merge": merge},
                "gpu_launches": args.steps * kernels_per_step,
                "pct_of_peak": round(100 * gbs / world / peak, 2),
                "peak_source": "%s (%.0f GB/s)" % (peak_src, peak),
                "per_rank_ms_per_step": [round(x, 5) for x in rank_ms],
                "cold_ms": round(cold_ms, 5) if cold_ms is not None else None,
                "cold_pct_of_peak": (round(100 * nbytes / (cold_ms * 1e-3) / 1e9 / peak, 2)
                                     if cold_ms is not None else None),
                "clocks": clk.summary()}), flush=True)
        return

    # end to end through the public API with the step's inputs and output in
    # page-locked host memory: paged_gqa_decode_host, whose kernel reads q, the
    # block table and the lengths over the host link and writes out back the
    # same way, so no separate copy is enqueued.  The KV pool is the resident
    # cache and stays in HBM.
    h_q = w.q.cpu().pin_memory()
    h_bt = w.block_table.cpu().pin_memory()
    h_sl = w.seq_lens.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ws_h = torch.zeros(max(256, pgd.paged_gqa_workspace_size_host(pool, w.B, 1, w.Hq,
                                                                  h_bt.shape[1])),
                       dtype=torch.uint8, device=dev)

    def e2e_step():
        pgd.paged_gqa_decode_host(pool, h_q, h_bt, h_sl, w.scale, out=h_out, workspace=ws_h,
                                  stream=stream)

    # the same step with the inputs copied in and the output copied back by
    # cudaMemcpyAsync around the device-memory call, for comparison
    d_q, d_bt, d_sl = torch.empty_like(w.q), torch.empty_like(w.block_table), torch.empty_like(
        w.seq_lens)

    def copy_step():
        d_q.copy_(h_q, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        pgd.paged_gqa_decode(pool, d_q, d_bt, d_sl, w.scale, out=out, workspace=ws, stream=stream)
        h_out.copy_(out, non_blocking=True)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    e2e_ms = timed(e2e_step)
    e2e_out = h_out.clone()
    copy_ms = timed(copy_step)
    if not torch.equal(e2e_out, h_out):   # h_out now holds the device-memory call's result
        raise RuntimeError("paged_gqa_decode_host result differs from paged_gqa_decode")
    status = pgd.paged_gqa_get_error(pool, stream)
    if status != 0:
        raise RuntimeError("device error: %s" % pgd.strerror(status))
    h2d = (w.q.numel() * w.q.element_size() + w.block_table.numel() * 4 + w.seq_lens.numel() * 4)
    d2h = out.numel() * out.element_size()

    if rank != 0:
        return
    peak, peak_src = peak_hbm()
    value = whole_job_gbs(nbytes, t_ms, world)
    per_gpu = nbytes / (t_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": describe(w), "parallelism": "replicas x%d" % world,
                   "l2": "no flush: each step streams %.0f MB of K/V, above the 126 MB L2"
                         % (nbytes / 1e6),
                   "launch": launch_note(args),
                   "algorithmic_bytes_per_step": nbytes, "merge": merge},
        "pct_of_peak": round(100 * per_gpu / peak, 2),
        "pct_of_nominal_8tbs": round(100 * per_gpu / NOMINAL_HBM_GBS, 2),
        "peak_source": "%s (%.0f GB/s)" % (peak_src, peak),
        "tokens_per_s_per_layer": round(world * w.B / (t_ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(per_gpu, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(per_gpu / peak, 4), "traffic": ncu_traffic(args.config),
                     "note": "achieved = algorithmic bytes / event-timed step: the decode "
                             "kernel, plus the run-merge kernel when the plan merges split runs "
                             "separately (config.merge = separate), so a lower bound on the "
                             "decode kernel's own rate"},
        "per_rank_ms_per_step": [round(x, 5) for x in rank_ms],
        "e2e": {"value": round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "path": "paged_gqa_decode_host, page-locked host q / block table / lengths / "
                        "out used in place by the kernel, one launch per step (this entry keeps "
                        "the split-run merge inside the decode kernel)",
                "copy_path_ms_per_step": round(copy_ms, 5),
                "copy_path": "cudaMemcpyAsync of the three inputs, paged_gqa_decode, "
                             "cudaMemcpyAsync of out"},
        "gpu_launches": args.steps * kernels_per_step,
        "clocks": clk.summary(),
    }
    if cold_ms is not None:
        cold = nbytes / (cold_ms * 1e-3) / 1e9
        line["roofline"].update({
            "cold_ms": round(cold_ms, 5), "cold_achieved": round(cold, 2),
            "cold_frac": round(cold / peak, 4),
            "cold_note": "median of %d single steps, each after a read of a buffer "
                         "twice the L2 size on the same stream; events around the step alone"
                         % args.cold_reps})
    if not args.no_cpu_baseline and world == 1:
        rate, sample, cores, _ = cpu_oracle_rate(w, args.cpu_seconds, args.cpu_threads)
        line["cpu_baseline"] = {"value": round(rate, 4), "unit": "GB/s", "cores": cores,
                                "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="llama3_8b", choices=sorted(gen.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host cores the CPU oracle runs on (cpu_baseline and --impl "
                         "reference); 0 = all")
    ap.add_argument("--op", default="decode", choices=["decode", "decode_ex", "append"],
                    help="decode (the headline), decode_ex (several query tokens and/or a "
                         "window), append (KV write path)")
    ap.add_argument("--q-len", type=int, default=4)
    ap.add_argument("--window", type=int, default=0)
    ap.add_argument("--launch", default="graph", choices=["graph", "stream"],
                    help="timed steps replayed as one CUDA graph (default) or launched one "
                         "by one from Python")
    ap.add_argument("--cold-reps", type=int, default=50,
                    help="single launches after an L2 flush for the cold figure (0: skip)")
    ap.add_argument("--profile", action="store_true",
                    help="only W + K step launches (for ncu); prints no bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # no launcher: start one rank per GPU of this node under torch.distributed.run
        sys.exit(subprocess.call(relaunch_cmd(sys.argv[1:], args.gpus, free_port())))
    world, rank, local = dist_setup()
    if world != args.gpus:
        print("bench.py: --gpus %d but the launcher started %d rank(s)" % (args.gpus, world),
              file=sys.stderr)
        sys.exit(2)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
