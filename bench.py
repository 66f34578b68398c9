"""Decode-step benchmark: tok/s and HBM roofline fraction of the block-quantized decode step.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one decode step of every sequence of the workload (embedding, all
layers, LM head, greedy argmax), replayed as one CUDA graph with tokens and
positions chained on the device.  Timed: K steps after W warm-up steps, CUDA
events on the launching stream, barrier + synchronize on both sides, max over
ranks.  With N > 1 (torchrun) every rank runs an independent replica ("weak"
scaling; the step has no exchange between GPUs).

--impl reference times the float64 CPU oracle on the same workload (a bounded
sample of steps) on the host cores and prints the same JSON line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode tok/s per step and achieved HBM GB/s vs 8 TB/s roofline (Q8_0/Q4_0)"
BPB = {"q8_0": 34, "q4_0": 18}
NOMINAL_HBM_GBS = 8000.0  # the 8 TB/s roofline the metric names
DEFAULT_WORKLOAD = "llama3_8b_q8_b16"  # the largest single-GPU workload, one of the two the 70 % target names


# ----------------------------------------------------------------------------------------------
# algorithmic bytes (each weight byte once per step, KV rows read once, outputs written once)
# ----------------------------------------------------------------------------------------------
def matrix_bytes(s: synth.ModelShape) -> dict[str, float]:
    """GGUF bytes of each GEMV's weights: one layer's fused Q/K/V, Wo, gate/up and down, and the head."""
    bpb = BPB[s.w_type] / 32.0
    D, qd, kvd, F, V = s.dim, s.qd, s.kvd, s.ffn_dim, s.vocab
    return {"qkv": (qd + 2 * kvd) * D * bpb, "wo": D * qd * bpb, "gateup": 2 * F * D * bpb, "down": D * F * bpb,
            "head": V * D * bpb}


def stage_bytes(wl: synth.Workload, pos: np.ndarray) -> dict[str, float]:
    s = wl.shape
    bpb = BPB[s.w_type] / 32.0
    B = wl.batch
    D, qd, kvd, F, V = s.dim, s.qd, s.kvd, s.ffn_dim, s.vocab
    w = matrix_bytes(s)
    attn_rows = float(np.sum(pos + 1))
    if wl.kv_type == "q8_0":
        # per row and side kvd / 32 blocks of 34 bytes; the new rows go through fp32 staging (written by the
        # QKV GEMV, read by the quantiser) before their blocks are written
        kv_row, kv_new = kvd / 32 * 34, kvd * 4 * 2 + kvd / 32 * 34
    else:
        kv_row, kv_new = kvd * 2, kvd * 2
    return {
        "embed": B * D * (2.0 if not s.tied else bpb) + B * D * 4,
        "qkv": w["qkv"] + B * (D * 4 + qd * 4 + 2 * kv_new) + D * 4,
        "attn": attn_rows * kv_row * 2 + B * qd * 4 * 2,
        "wo": w["wo"] + B * (qd * 4 + 2 * D * 4),
        "gateup": w["gateup"] + B * (D * 4 + F * 4) + D * 4,
        "down": w["down"] + B * (F * 4 + 2 * D * 4),
        "head": w["head"] + B * (D * 4 + V * 4) + D * 4,
    }


def step_bytes(wl: synth.Workload, pos: np.ndarray) -> float:
    b = stage_bytes(wl, pos)
    L = wl.shape.n_layers
    return b["embed"] + L * (b["qkv"] + b["attn"] + b["wo"] + b["gateup"] + b["down"]) + b["head"]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# sources each measured kernel is compiled from
KERNEL_SOURCES = {
    "step_kernel": ("common.cuh", "gemv_core.cuh", "internal.h", "kernels_step.cuh", "kernels_step_q4.cu",
                    "kernels_step_q8.cu", "layout.cuh"),
    "attn": ("common.cuh", "internal.h", "kernels_attn.cu"),
}
STEP_KERNEL_SOURCES = KERNEL_SOURCES["step_kernel"]

# DRAM bytes per launch of a kernel from one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum),
# keyed by (workload, kernel) with a hash of that kernel's sources at the capture: a changed kernel
# reports no traffic until it is captured again.  Captures of a cut model (fewer layers) are per launch
# of the same kernel on the same per-layer shapes.
KERNEL_TRAFFIC = {
    # step_kernel<Q8_0, 64, 3> / <Q4_0, 128, 1>, 4th launch of `bench.py --workload smollm_q8 | llama2_7b_q4
    # --steps 4 --warmup 3 --no-cpu-baseline` (full size, one pass)
    ("smollm_q8", "step_kernel"): ("3ef517f4638baae0", 190925824 + 3020032),
    ("llama2_7b_q4", "step_kernel"): ("3ef517f4638baae0", 5866404352 + 9216768),
    # attn_tc_kernel<128, 4, fp16 / Q8_0 cache>, 4th launch of `bench.py [--workload llama3_8b_q8_b16_kvq8]
    # --layers 1 --steps 1 --warmup 3 --no-cpu-baseline` (one layer: the per-layer shape of the full model)
    ("llama3_8b_q8_b16", "attn"): ("90937cb4d8f6371e", 537818880 + 9653504),
    ("llama3_8b_q8_b16_kvq8", "attn"): ("90937cb4d8f6371e", 291743232 + 9249024),
}


def csrc_hash(files=STEP_KERNEL_SOURCES) -> str:
    """Hash of the step kernel's sources (and the C ABI header) with comments and blank space removed."""
    import hashlib
    import re
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_quantized_token_gb300", "csrc")
    paths = [os.path.join(d, f) for f in files] + [os.path.join(ROOT, "include", "er.h")]
    for path in paths:
        with open(path) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(os.path.basename(path).encode() + b"\0" + " ".join(src.split()).encode())
    return h.hexdigest()[:16]


def kernel_traffic(workload: str, kernel: str = "step_kernel"):
    e = KERNEL_TRAFFIC.get((workload, kernel))
    return e[1] if e and e[0] == csrc_hash(KERNEL_SOURCES[kernel]) else None


def max_over_ranks(value: float, device) -> float:
    """Largest value over the ranks of the default process group (the value itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------------------------
def run_ours(args, rank: int, world: int, local_rank: int) -> dict | None:
    import torch

    from block_quantized_token_gb300 import build as libbuild
    if rank == 0 and not libbuild.up_to_date():
        libbuild.build()  # one rank builds; the others wait for it below
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    from block_quantized_token_gb300 import er, runtime

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.workload(args.workload)
    s = wl.shape
    B = wl.batch
    K, W = args.steps, args.warmup
    cap = wl.prefill + max(K, W, 1)
    wl_run = wl.with_(steps=cap - wl.prefill)

    t0 = time.time()
    threads = min(32, os.cpu_count() or 1)
    model = runtime.DecodeModel(s, synth.model_weights(s, threads=threads), max_batch=B)
    state = runtime.DecodeState(model, B, cap, kv_type=wl.kv_type)
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=threads) as ex:  # draws run in parallel, writes in order
        jobs = [(b, l) for b in range(B) for l in range(s.n_layers)]
        for (b, l), (k, v) in zip(jobs, ex.map(lambda bl: synth.kv_prefill(wl_run, *bl), jobs)):
            state.write_rows(b, l, k, v)
    setup_s = time.time() - t0

    if args.schedule != "auto":
        state.set_schedule({"persistent": er.ER_SCHEDULE_PERSISTENT, "kernels": er.ER_SCHEDULE_KERNELS}[args.schedule])
    schedule = {er.ER_SCHEDULE_PERSISTENT: "persistent", er.ER_SCHEDULE_KERNELS: "kernels"}[state.schedule]
    launches_step = er.er_kv_launches_per_step(state.handle)

    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    pos = torch.empty(B, dtype=torch.int32, device=dev)
    logits = torch.empty((B, s.vocab), dtype=torch.float32, device=dev)

    def reset():
        tok.copy_(torch.from_numpy(wl.tokens0()))
        pos.copy_(torch.from_numpy(wl.positions0()))

    def one_step():
        er.er_decode_step(tok.data_ptr(), pos.data_ptr(), state.handle, logits.data_ptr(), tok.data_ptr(), sp)
        er.er_positions_increment(pos.data_ptr(), B, sp)

    with torch.cuda.stream(stream):
        reset()
        for _ in range(W):
            one_step()
        reset()
    stream.synchronize()

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    # events around every step graph (on the launching stream) give the step
    # kernel's own duration; the outer pair times the whole chain
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a read of 256 MiB (larger than L2) between steps leaves L2 holding only clean lines, so no
    # write-back of the flush itself lands inside the next step's timing
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev) if args.flush_l2 else None
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(K):
            if flush is not None:  # a read larger than L2 between steps (outside the per-step events)
                flush.sum()
            evs[i][0].record(stream)
            er.er_decode_step(tok.data_ptr(), pos.data_ptr(), state.handle, logits.data_ptr(), tok.data_ptr(), sp)
            evs[i][1].record(stream)
            er.er_positions_increment(pos.data_ptr(), B, sp)
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    graph_ms = [a.elapsed_time(b) for a, b in evs]
    # with the flush, the step time is the sum of the step graphs alone
    ms = sum(graph_ms) if flush is not None else ev0.elapsed_time(ev1)
    clock_info = clocks.stop() if rank == 0 else None
    ms = max_over_ranks(ms, dev)
    st, code, nf = state.device_error()
    if code:
        raise RuntimeError(f"device error flags {code}")

    # ---- end to end through the C ABI with host buffers (pinned), one H2D + D2H per step
    tok_h = torch.from_numpy(wl.tokens0()).pin_memory()
    pos_h = torch.from_numpy(wl.positions0()).pin_memory()
    out_h = torch.empty(B, dtype=torch.int32).pin_memory()
    argmax_d = torch.empty(B, dtype=torch.int32, device=dev)

    def e2e_step():
        tok.copy_(tok_h, non_blocking=True)
        pos.copy_(pos_h, non_blocking=True)
        er.er_decode_step(tok.data_ptr(), pos.data_ptr(), state.handle, logits.data_ptr(), argmax_d.data_ptr(), sp)
        out_h.copy_(argmax_d, non_blocking=True)
        stream.synchronize()
        tok_h.copy_(out_h)
        pos_h.add_(1)

    with torch.cuda.stream(stream):
        for _ in range(min(W, 3)):
            e2e_step()
        tok_h.copy_(torch.from_numpy(wl.tokens0()))
        pos_h.copy_(torch.from_numpy(wl.positions0()))
        torch.cuda.synchronize(dev)
        e0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        e2e_s = time.perf_counter() - e0
    e2e_s = max_over_ranks(e2e_s, dev)

    positions = wl.positions0()[None, :] + np.arange(K)[:, None]
    per_step_bytes = [step_bytes(wl, p) for p in positions]
    bytes_step = float(np.mean(per_step_bytes))

    # ---- roofline of the dominant kernel
    roof = None
    if rank == 0:
        peaks = measured_peaks()
        if schedule == "persistent":
            # one launch per step: the step kernel is the whole step (plus a 4-byte memset in the same graph)
            launch_ms = float(np.mean(graph_ms))
            achieved = bytes_step / (launch_ms / 1e3) / 1e9
            roof = {"bound": "hbm", "kernel": "step_kernel", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                    "traffic": kernel_traffic(wl.name),
                    "peak_source": f"{peaks['source']} hbm_gbs (STREAM-style copy)",
                    "bytes_per_launch": bytes_step, "us_per_launch": launch_ms * 1e3,
                    "timing": "CUDA events around each step graph inside the timed region"}
        else:
            roof = stage_roofline(er, state, wl, tok, pos, logits, stream, dev)

    tokens = B * K * world
    result = None
    if rank == 0:
        result = {
            "metric": METRIC,
            "value": tokens / (ms / 1e3),
            "unit": "tok/s",
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": ms / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "model": f"{s.n_layers}L d{s.dim} {s.n_heads}/{s.n_kv_heads}x{s.head_dim} "
                                                     f"ffn{s.ffn_dim} V{s.vocab} {s.w_type} "
                                                     f"{'tied' if s.tied else 'untied'}",
                       "batch": B, "context": wl.prefill, "kv_cache": wl.kv_type, "chained_steps": K, "schedule": schedule,
                       "step_bytes": bytes_step, "step_gbs": bytes_step / (ms / K / 1e3) / 1e9,
                       "step_roofline_frac": bytes_step / (ms / K / 1e3) / 1e9 / measured_peaks()["hbm_gbs"],
                       "step_frac_of_8tbs": bytes_step / (ms / K / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                       "l2": ("L2 flushed between steps (a 256 MiB read), step graphs timed alone" if args.flush_l2
                              else "inputs larger than L2" if bytes_step > 129e6
                              else "L2-resident working set, not flushed"),
                       "parallelism": f"replicas x{world}", "setup_s": round(setup_s, 1)},
            "e2e": {"value": tokens / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": 8 * B, "d2h_bytes_per_step": 4 * B},
            "gpu_launches": (launches_step + 1) * K,
            "roofline": roof,
            "clocks": clock_info,
        }
    state.close()
    model.close()
    return result


def stage_roofline(er, state, wl, tok, pos, logits, stream, dev, iters: int = 20) -> dict:
    """Average event-timed duration of each stage kernel at the workload's first position.

    Every launch is preceded by a read of a 256 MiB buffer (larger than L2), so
    the weights come from HBM as in the chained step.  A read, not a write: a
    written buffer would leave up to an L2's worth of dirty lines whose
    write-back lands inside the timed launch.  Returns the roofline of the
    stage with the largest total time per step.
    """
    import torch
    peaks = measured_peaks()
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    pos_np = wl.positions0()
    sb = stage_bytes(wl, pos_np)
    L = wl.shape.n_layers
    per_step = {"qkv": L, "attn": L, "wo": L, "gateup": L, "down": L, "head": 1}
    ids = {"qkv": er.ER_STAGE_QKV, "attn": er.ER_STAGE_ATTN, "wo": er.ER_STAGE_WO, "gateup": er.ER_STAGE_GATEUP,
           "down": er.ER_STAGE_DOWN, "head": er.ER_STAGE_HEAD}
    sp = stream.cuda_stream
    durs = {}
    with torch.cuda.stream(stream):
        tok.copy_(torch.from_numpy(wl.tokens0()))
        pos.copy_(torch.from_numpy(pos_np))
        for name, sid in ids.items():
            tot = 0.0
            for i in range(iters + 2):
                flush.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                er.er_launch_stage(state.handle, sid, L // 2, tok.data_ptr(), pos.data_ptr(), logits.data_ptr(),
                                   None, sp)
                e1.record(stream)
                e1.synchronize()
                if i >= 2:
                    tot += e0.elapsed_time(e1)
            durs[name] = tot / iters
    share = {n: durs[n] * per_step[n] for n in durs}
    top = max(share, key=share.get)
    achieved = sb[top] / (durs[top] / 1e3) / 1e9
    return {"bound": "hbm", "kernel": top, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
            "traffic": kernel_traffic(wl.name, top) if top in KERNEL_SOURCES else None,
            "peak_source": f"{peaks['source']} hbm_gbs (burst, kernel timed alone)",
            "bytes_per_launch": sb[top], "us_per_launch": durs[top] * 1e3,
            "stages_us": {n: round(d * 1e3, 2) for n, d in durs.items()},
            "stages_gbs": {n: round(sb[n] / (durs[n] / 1e3) / 1e9, 1) for n in durs}}


# ----------------------------------------------------------------------------------------------
# the oracle arm (CPU, float64)
# ----------------------------------------------------------------------------------------------
def _oracle_run(wl: synth.Workload, n_layers: int, steps: int, budget_s: float, seqs) -> tuple[float, int]:
    """Seconds per step of the oracle on the workload cut to `n_layers` layers (inputs drawn before timing)."""
    import dataclasses

    import oracle
    s = dataclasses.replace(wl.shape, n_layers=n_layers)
    wk = wl.with_(shape=s)
    tensors = synth.model_weights(s)
    ocfg = oracle.OracleConfig(**{k: getattr(s, k) for k in oracle.OracleConfig.__dataclass_fields__})
    cache = oracle.OracleCache(ocfg, wl.batch, wl.prefill + steps, kv_type=wl.kv_type)
    for b in seqs:
        for l in range(n_layers):
            k, v = synth.kv_prefill(wk, b, l)
            cache.fill(b, l, k, v)
    model = oracle.OracleModel(ocfg, tensors)
    tok, pos = wl.tokens0().astype(np.int64), wl.positions0().astype(np.int64)
    done = 0
    t0 = time.perf_counter()
    for _ in range(steps):
        _, am, _ = oracle.decode_step(model, cache, tok, pos, seqs=seqs)
        tok[seqs] = am
        pos[seqs] += 1
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return (time.perf_counter() - t0) / done, done


def oracle_sample(wl: synth.Workload, steps: int, budget_s: float, seqs=None) -> tuple[float, int, dict]:
    """Time the oracle (as it stands) on consecutive steps of the workload; returns (tok/s, steps, info).

    The weights and the prefilled cache are drawn before the clock starts.  When
    a whole-model step would not fit the budget, the oracle runs the model cut
    to 1 and to 2 layers, and the step time is extrapolated linearly in the
    layer count (embedding and head are the intercept), which info says.
    """
    seqs = [0] if seqs is None else seqs
    L = wl.shape.n_layers
    t1, _ = _oracle_run(wl, 1, 1, budget_s, seqs)
    if t1 * L * 1.2 <= budget_s:
        per, done = _oracle_run(wl, L, steps, budget_s, seqs)
        return len(seqs) / per, done, {"seconds": per * done, "how": f"{done} consecutive steps of the whole model"}
    per1, d1 = _oracle_run(wl, 1, 2, budget_s / 2, seqs)
    per2, d2 = _oracle_run(wl, 2, 2, budget_s / 2, seqs)
    slope = max(per2 - per1, 1e-9)
    per = per1 + (L - 1) * slope
    return len(seqs) / per, d1 + d2, {
        "seconds": per1 * d1 + per2 * d2,
        "how": f"{d1} + {d2} steps of the model cut to 1 and 2 layers, step time extrapolated linearly to {L} layers "
               f"({per:.1f} s/step)"}


def gemv_sweep(reps: int = 50) -> dict:
    """The isolated Q4_0 GEMV sweep of the 135M-shaped Q4_0 workload: M x K = 576x576, 1536x576, 49152x576,
    batch 1, through er_matrix_gemv.  Each launch follows a 256 MiB read (larger than L2), so the weights come
    from HBM; CUDA events around each launch on the launching stream."""
    import torch
    from block_quantized_token_gb300 import build as libbuild
    if not libbuild.up_to_date():
        libbuild.build()
    from block_quantized_token_gb300 import er
    peaks = measured_peaks()
    flush = torch.ones(64 << 20, dtype=torch.float32, device="cuda")  # read, not written: no dirty lines
    stream = torch.cuda.Stream()
    out = {}
    for rows, cols in ((576, 576), (1536, 576), (49152, 576)):
        rng = np.random.default_rng(rows)
        raw = synth.quantize((0.02 * rng.standard_normal((rows, cols))).astype(np.float32), "q4_0")
        dev = torch.from_numpy(raw).cuda()
        m = er.er_matrix_create(er.DTYPES["q4_0"], rows, cols, dev.data_ptr())
        x = torch.from_numpy(rng.standard_normal((1, cols)).astype(np.float32)).cuda()
        y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
        tot = 0.0
        with torch.cuda.stream(stream):
            for i in range(reps + 3):
                flush.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                er.er_matrix_gemv(m, x.data_ptr(), 1, y.data_ptr(), stream.cuda_stream)
                e1.record(stream)
                e1.synchronize()
                if i >= 3:
                    tot += e0.elapsed_time(e1)
        er.er_matrix_destroy(m)
        us = tot / reps * 1e3
        nbytes = rows * cols // 32 * 18 + cols * 4 + rows * 4
        out[f"{rows}x{cols}"] = {"us": round(us, 2), "bytes": nbytes, "gbs": round(nbytes / us / 1e3, 1),
                                 "frac": round(nbytes / us / 1e3 / peaks["hbm_gbs"], 4)}
    return out


def run_prefill(args) -> dict:
    """Chunked prefill of `args.prefill` seeded tokens into one sequence of the workload's model (a fresh
    cache from position 0), timed with CUDA events over `args.steps` repetitions after `args.warmup`."""
    import torch

    from block_quantized_token_gb300 import build as libbuild
    if not libbuild.up_to_date():
        libbuild.build()
    from block_quantized_token_gb300 import runtime
    wl = synth.workload(args.workload)
    s = wl.shape
    n = args.prefill
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    threads = min(32, os.cpu_count() or 1)
    model = runtime.DecodeModel(s, synth.model_weights(s, threads=threads), max_batch=1)
    state = runtime.DecodeState(model, 1, n, kv_type=wl.kv_type)
    toks = torch.tensor(np.random.default_rng(1).integers(0, s.vocab, n).astype(np.int32), device=dev)
    logits = torch.empty(s.vocab, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    for _ in range(args.warmup):
        state.prefill(0, toks, 0, logits, stream=stream.cuda_stream)
    stream.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            state.prefill(0, toks, 0, logits, stream=stream.cuda_stream)
            b.record(stream)
    torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    if state.device_error()[1]:
        raise RuntimeError("device error flags after prefill")
    # algorithmic bytes: every chunk of 16 reads the layers' weights once and the K/V rows below its last
    # position once, and writes its rows; the head once for the last token
    w = matrix_bytes(s)
    per_layer_w = w["qkv"] + w["wo"] + w["gateup"] + w["down"]
    kv_row = s.kvd / 32 * 34 if wl.kv_type == "q8_0" else s.kvd * 2
    chunks = (n + 15) // 16
    rows_read = sum(min(n, 16 * (c + 1)) for c in range(chunks))
    nbytes = chunks * s.n_layers * per_layer_w + w["head"] + s.n_layers * 2 * kv_row * (rows_read + n)
    gbs = nbytes / (ms / 1e3) / 1e9
    peaks = measured_peaks()
    state.close()
    model.close()
    return {"metric": "prefill tok/s (chunks of 16 tokens through the batched decode kernels)", "value": n / (ms / 1e3),
            "unit": "tok/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_prefill": ms,
            "higher_is_better": True, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "prompt_tokens": n, "kv_cache": wl.kv_type, "chunk": 16},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
                         "bytes_per_prefill": nbytes},
            "clocks": clock_info}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed chained steps (default: the workload's chain)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--flush-l2", action="store_true",
                    help="read 256 MiB between steps and time the step graphs alone (for L2-sized workloads)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--gemv-sweep", action="store_true",
                    help="time the isolated Q4_0 GEMV sweep (576x576, 1536x576, 49152x576) and print it")
    ap.add_argument("--schedule", default="auto", choices=["auto", "persistent", "kernels"],
                    help="step schedule (auto: the persistent kernel where the shape allows it)")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the layer count (smaller cases for profiling; not a bench workload)")
    ap.add_argument("--prefill", type=int, default=None,
                    help="time er_prefill of this many tokens into one sequence of the workload's model instead")
    args = ap.parse_args()

    if args.gemv_sweep:
        print(json.dumps({"gemv_sweep_q4_0": gemv_sweep(), "unit": "us per launch, algorithmic GB/s",
                          "peak_gbs": measured_peaks()["hbm_gbs"]}))
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = synth.workload(args.workload)
    if args.steps is None:
        args.steps = wl.steps
    if args.layers:
        import dataclasses
        wl = wl.with_(name=f"{wl.name}_L{args.layers}", shape=dataclasses.replace(wl.shape, n_layers=args.layers))
        synth.WORKLOADS[wl.name] = wl
        args.workload = wl.name
    cores = os.cpu_count()

    if args.impl == "reference":
        if rank != 0:
            return
        budget = max(10.0, min(60.0, args.cpu_budget * 2))
        tps, done, info = oracle_sample(wl, args.steps, budget, seqs=[0])
        sample = f"sequence 0 from position {wl.prefill}: {info['how']}"
        line = {"metric": METRIC, "value": tps, "unit": "tok/s", "n_gpus": args.gpus, "steps": done,
                "warmup": 0, "ms_per_step": info["seconds"] * 1e3 / max(done, 1), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": wl.name, "batch": wl.batch, "context": wl.prefill, "kv_cache": wl.kv_type},
                "impl": "reference",
                "cpu_baseline": {"value": tps, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample},
                "e2e": {"value": tps, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.prefill:
        if rank == 0:
            print(json.dumps(run_prefill(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if args.no_cpu_baseline:
            res["cpu_baseline"] = None
        else:
            tps, done, info = oracle_sample(wl, 64, args.cpu_budget, seqs=[0])
            res["cpu_baseline"] = {"value": tps, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                   "sample": f"sequence 0 from position {wl.prefill}: {info['how']} "
                                             f"({info['seconds']:.1f} s timed, numpy float64, BLAS on all cores)"}
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
