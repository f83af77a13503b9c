"""Benchmark: fused RNN training step (forward_training + backward_data +
backward_weights) on the Deep Speech 2 LSTM layer shape, 1 GPU per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ds2_lstm]
                    [--impl ours|reference]

One JSON line on rank 0.  A step is one pass of the whole hot path over one
batch (N=20 sequences of T=300) with inputs resident in HBM; L2 is flushed
(256 MiB write, untimed) before every timed step; each step is bracketed by
CUDA events on the launching stream.  Under torchrun the ranks run data
parallel over the batch: each rank takes its own N sequences (weak scaling)
and the step ends with one all-reduce (sum) of the weight gradients
(layer_rnn_gb300.dp); value = sequences of all ranks / max-over-ranks step
time.

``--impl reference`` times the float64 CPU oracle (the only other
implementation) on a bounded sample of the same workload on the host cores.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from layer_rnn_gb300 import workloads as wl  # noqa: E402

METRIC = "LSTM/GRU fwd+bwd sequences/s and effective TFLOP/s at DS2 shape, 1×GB300"
PHASE_NAMES = ("input_gemm", "rec_fwd", "rec_bwd", "dx_gemm", "dw_gemm")
PHASE_KERNELS = {"input_gemm": "gemm_tc_kernel (+ absmax, split_f16): input projection",
                 "rec_fwd": "rec_fwd_* persistent recurrent forward",
                 "rec_bwd": "rec_bwd_* persistent recurrent backward",
                 "dx_gemm": "gemm_tc_kernel (+ absmax, split_f16): dX",
                 "dw_gemm": "gemm_tc_kernel (+ absmax, split_f16 / transpose, splitk_reduce, "
                            "colsum): dW, db"}


def gates(mode):
    return wl.GATES[mode]


def phase_flops(cfg):
    """Algorithmic flops per phase for one training step (whole stack)."""
    G, H, T, N, D = gates(cfg["mode"]), cfg["H"], cfg["T"], cfg["N"], wl.num_directions(cfg)
    out = dict.fromkeys(PHASE_NAMES, 0.0)
    for l in range(cfg["L"]):
        I_l = cfg["I"] if l == 0 else D * H
        per = 2.0 * T * N * G * H
        out["input_gemm"] += D * per * I_l
        out["rec_fwd"] += D * per * H
        out["rec_bwd"] += D * per * H
        out["dx_gemm"] += D * per * I_l
        out["dw_gemm"] += D * per * (I_l + H)
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


def include_closure(src):
    """The source file and every header it includes with #include "...",
    transitively, resolved against the including file's folder; sorted by path
    after the source itself."""
    import re
    pat = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)
    first = os.path.normpath(os.path.join(ROOT, src))
    seen, todo = {first}, [first]
    while todo:
        fn = todo.pop()
        with open(fn) as f:
            text = f.read()
        for inc in pat.findall(text):
            p = os.path.normpath(os.path.join(os.path.dirname(fn), inc))
            if os.path.exists(p) and p not in seen:
                seen.add(p)
                todo.append(p)
    return [first] + sorted(seen - {first})


def kernel_source_sha256(src):
    """sha256 over a kernel's source file and the headers it includes,
    transitively: a change to any of them can change the kernel, a change to
    another part's header cannot."""
    import hashlib
    h = hashlib.sha256()
    for fn in include_closure(src):
        h.update(os.path.relpath(fn, ROOT).encode() + b"\0")
        with open(fn, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_for(phase, cfg):
    """DRAM bytes per launch of the phase's kernel from a committed ncu summary,
    or None when there is none for this workload or the kernel source (or a
    header it may include) changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        doc = json.load(f)
    ent = doc.get(cfg["name"], {}).get(phase)
    if not ent or "sources_sha256" not in ent:
        return None
    if not os.path.exists(os.path.join(ROOT, ent["source"])):
        return None
    if kernel_source_sha256(ent["source"]) != ent["sources_sha256"]:
        return None
    return ent["dram_bytes_per_launch"]


def fp32_simt_peak_tflops(num_sms, sm_mhz):
    # 128 fp32 FMA lanes per SM per clock, 2 flop per FMA
    return num_sms * 128 * 2 * sm_mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ----------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# distributed plumbing (barrier and max over ranks; the data path's one
# collective, the dW all-reduce, is layer_rnn_gb300.dp)
# ----------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def max_over_ranks(value, dist, device="cpu"):
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def aggregate_sequences_per_s(n_per_rank, world_size, ms_step_max):
    """Whole-job throughput: the sequences every rank processed in one step
    over the slowest rank's step time (weak scaling: N per rank is fixed)."""
    return n_per_rank * world_size / (ms_step_max * 1e-3)


# ----------------------------------------------------------------------------
# the CPU oracle, timed (baseline / reference arm)
# ----------------------------------------------------------------------------
def time_oracle(cfg, budget_s=20.0, max_reps=3):
    """Oracle fwd+bwd on a prefix of the sequences (shorter T), scaled to full
    sequences.  Returns (sequences_per_s, sample description, seconds spent)."""
    import oracle
    T_full = cfg["T"]
    # probe on a short prefix, then grow within the budget
    T_s = max(1, min(T_full, 10))
    spent = 0.0
    best = None
    reps = 0
    while True:
        c = wl.with_sizes(cfg, T=T_s)
        inp = wl.make_inputs(c)
        t0 = time.perf_counter()
        oracle.run_flat(c["mode"], c["L"], c["bidir"], c["I"], c["H"], inp["x"], inp["h0"],
                        inp["c0"], inp["w"], inp["dy"], inp["dhy"], inp["dcy"])
        dt = time.perf_counter() - t0
        spent += dt
        reps += 1
        per_full_seq = dt * (T_full / T_s) / c["N"]
        best = per_full_seq if best is None else min(best, per_full_seq)
        if T_s < T_full and spent + dt * min(T_full / T_s, 4) * 1.5 < budget_s:
            T_s = min(T_full, T_s * 4)
            continue
        if reps < max_reps and spent + dt < budget_s:
            continue
        break
    sample = ("float64 oracle fwd+bwd on the first %d of %d time steps of the %s workload "
              "(N=%d sequences), best of %d runs, scaled by %d/%d to whole sequences"
              % (T_s, T_full, cfg["name"], cfg["N"], reps, T_full, T_s))
    return 1.0 / best, sample, spent


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, cfg):
    import torch
    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init("nccl")
    line = measure(args, cfg, dist, dev, rank, ws_n, local)
    if cfg["name"] == "ds2_lstm" and not args.no_gru:
        # the metric is LSTM/GRU at the DS2 shape: the GRU layer of the same
        # shape, timed the same way, rides along in the same line
        g = measure(args, wl.WORKLOADS["ds2_gru"], dist, dev, rank, ws_n, local)
        line["gru"] = {k: g[k] for k in ("value", "unit", "ms_per_step", "effective_tflops",
                                         "phases", "recurrent_paths", "roofline", "e2e",
                                         "varlen", "gpu_launches", "clocks")}
        line["gru"]["config"] = g["config"]
    if rank == 0 and not args.no_cpu_baseline:
        v, sample, spent = time_oracle(cfg, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "sequences/s",
                                "cores": os.cpu_count(), "kind": "oracle", "sample": sample,
                                "seconds": round(spent, 2)}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure(args, cfg, dist, dev, rank, ws_n, local):
    """Time one workload (device-resident steps, per-phase events, end to end
    through pinned host buffers) and return its bench line (no CPU baseline)."""
    import torch
    from layer_rnn_gb300 import binding as B
    from layer_rnn_gb300 import dp
    from layer_rnn_gb300 import tensors as tz
    T, N, I, H, L = cfg["T"], cfg["N"], cfg["I"], cfg["H"], cfg["L"]
    D = wl.num_directions(cfg)
    dt = cfg["dtype"]
    lstm = cfg["mode"] == "lstm"
    inp = wl.make_inputs(cfg, seed=cfg["seed"] + rank)
    r = B.Rnn(cfg["mode"], L, cfg["bidir"], I, H, dt, 0)
    paths = B.rnn_get_paths(r.h, N)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        x = tz.to_dev(inp["x"], dt, dev)
        h0 = tz.to_dev(inp["h0"], dt, dev)
        c0 = tz.to_dev(inp["c0"], "f32", dev) if lstm else None
        W = tz.to_dev(inp["w"], dt, dev)
        dy = tz.to_dev(inp["dy"], dt, dev)
        dhy = tz.to_dev(inp["dhy"], dt, dev)
        dcy = tz.to_dev(inp["dcy"], "f32", dev) if lstm else None
        y = tz.empty((T, N, D * H), dt, dev)
        hy = tz.empty((L * D, N, H), dt, dev)
        cy = tz.empty((L * D, N, H), "f32", dev) if lstm else None
        dx = tz.empty((T, N, I), dt, dev)
        dh0 = tz.empty((L * D, N, H), dt, dev)
        dc0 = tz.empty((L * D, N, H), "f32", dev) if lstm else None
        dW = tz.empty((inp["w"].size,), dt, dev)
        ws = r.alloc_workspace(T, N, dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream.synchronize()

    set0 = dict(x=x, h0=h0, c0=c0, W=W, dy=dy, dhy=dhy, dcy=dcy, y=y, hy=hy, cy=cy, dx=dx,
                dh0=dh0, dc0=dc0, dW=dW)

    def step_with(t):
        r.forward_training(t["x"], t["h0"], t["c0"], t["W"], t["y"], t["hy"], t["cy"], ws, stream)
        r.backward_data(t["W"], t["dy"], t["dhy"], t["dcy"], t["dx"], t["dh0"], t["dc0"], ws,
                        stream)
        r.backward_weights(t["x"], t["h0"], t["y"], ws, t["dW"], stream)
        if dist is not None:
            # data parallel over the batch: the one exchange, the sum of the
            # ranks' weight gradients (NCCL, on the launching stream)
            with torch.cuda.stream(stream):
                dp.allreduce_grads(t["dW"], dist)

    def step():
        step_with(set0)

    def timed(n, fn):
        evs = []
        for _ in range(n):
            with torch.cuda.stream(stream):
                flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        stream.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    # warm-up
    for _ in range(args.warmup):
        step()
    st = r.check_status(stream)
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)

    # device-resident timed region
    sampler = ClockSampler(local)
    barrier(dist)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.25)
    wall0 = time.perf_counter()
    ms = timed(args.steps, step)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(dist)
    clocks = sampler.stop()
    st = r.check_status(stream)
    if st != 0:
        raise RuntimeError("device status %d in timed region" % st)
    ms_step = statistics.mean(ms)
    ms_step_max = max_over_ranks(ms_step, dist, dev)

    # per-phase CUDA events on the launching stream (a second pass of K steps)
    B.rnn_enable_phase_timing(r.h, 1)
    ms2 = timed(args.steps, step)
    phases = B.rnn_get_phase_times(r.h)
    B.rnn_enable_phase_timing(r.h, 0)
    launches_per_step = sum(n for _, n in phases.values()) / args.steps

    # end to end: every step copies its inputs in from pinned host memory and
    # its results out to pinned host memory, as a training loop does: the
    # copies of step k+1's inputs and of step k-1's results run on two copy
    # streams under step k's compute (inputs and results double-buffered on
    # the device), and the K steps are timed as one region.  No L2 flush inside
    # it: a step's data (about 0.4 GB at DS2 sizes) is larger than L2.
    in_keys = ("x", "h0", "c0", "W", "dy", "dhy", "dcy")
    out_keys = ("y", "hy", "cy", "dx", "dh0", "dc0", "dW")
    pin = {}
    for k in in_keys:
        if set0[k] is not None:
            pin[k] = torch.empty(set0[k].shape, dtype=set0[k].dtype, pin_memory=True)
            pin[k].copy_(set0[k])
    pout = {k: torch.empty(set0[k].shape, dtype=set0[k].dtype, pin_memory=True)
            for k in out_keys if set0[k] is not None}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in pout.values())
    with torch.cuda.stream(stream):
        set1 = {k: (torch.empty_like(v) if v is not None else None) for k, v in set0.items()}
    sets = (set0, set1)
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    def e2e_run(K):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s_in.wait_event(start)
        done, copied = [None] * K, [None] * K
        for k in range(K):
            t = sets[k % 2]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(done[k - 2])      # step k-2 has read these inputs
                for key, h in pin.items():
                    t[key].copy_(h, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            stream.wait_event(ready)
            if k >= 2:
                stream.wait_event(copied[k - 2])      # step k-2's results are out
            step_with(t)
            done[k] = torch.cuda.Event()
            done[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[k])
                for key, h in pout.items():
                    h.copy_(t[key], non_blocking=True)
                copied[k] = torch.cuda.Event()
                copied[k].record(s_out)
        stream.wait_event(copied[K - 1])
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / K

    e2e_run(2)  # warm-up: the second buffer set and the copy streams
    barrier(dist)
    ms_e2e = e2e_run(args.steps)
    ms_e2e_max = max_over_ranks(ms_e2e, dist, dev)

    # the same batch padded to T with per-sequence lengths (the *_varlen
    # calls), device-resident like the main line
    lens_np = wl.make_lengths(cfg, seed=cfg["seed"] + rank)
    lens = torch.tensor(lens_np, dtype=torch.int32, device=dev)
    vpaths = B.rnn_get_paths_varlen(r.h, N)

    def step_varlen():
        r.forward_training_varlen(lens, x, h0, c0, W, y, hy, cy, ws, stream)
        r.backward_data_varlen(lens, W, dy, dhy, dcy, dx, dh0, dc0, ws, stream)
        r.backward_weights(x, h0, y, ws, dW, stream)
        if dist is not None:
            with torch.cuda.stream(stream):
                dp.allreduce_grads(dW, dist)

    for _ in range(args.warmup):
        step_varlen()
    barrier(dist)
    ms_var = statistics.mean(timed(args.steps, step_varlen))
    ms_var_max = max_over_ranks(ms_var, dist, dev)
    st = r.check_status(stream)
    if st != 0:
        raise RuntimeError("device status %d in the varlen steps" % st)

    # stacks: the same batch with inter-layer dropout (the *_dropout calls)
    drop = None
    if L > 1:
        p_drop = 0.3
        masks = torch.tensor(wl.make_dropout_masks(cfg, p_drop, seed=cfg["seed"] + rank),
                             device=dev)

        def step_dropout():
            r.forward_training_dropout(p_drop, masks, x, h0, c0, W, y, hy, cy, ws, stream)
            r.backward_data_dropout(p_drop, masks, W, dy, dhy, dcy, dx, dh0, dc0, ws, stream)
            r.backward_weights(x, h0, y, ws, dW, stream)
            if dist is not None:
                with torch.cuda.stream(stream):
                    dp.allreduce_grads(dW, dist)

        for _ in range(args.warmup):
            step_dropout()
        barrier(dist)
        ms_drop = max_over_ranks(statistics.mean(timed(args.steps, step_dropout)), dist, dev)
        st = r.check_status(stream)
        if st != 0:
            raise RuntimeError("device status %d in the dropout steps" % st)
        drop = {"value": round(aggregate_sequences_per_s(N, ws_n, ms_drop), 2),
                "unit": "sequences/s", "ms_per_step": round(ms_drop, 4), "p": p_drop,
                "calls": "rnn_forward_training_dropout + rnn_backward_data_dropout + "
                         "rnn_backward_weights, seeded Bernoulli masks, L2 flushed before "
                         "every step"}
    # the step protocol of the tensor-core recurrent forward alone (exchange
    # words written and polled, cluster barrier; no work): the term of the
    # recurrence's latency bound that no arithmetic removes
    empty_us = None
    if paths[0] == "tensor":
        try:
            empty_us = B.rnn_measure_step_protocol(r.h, stream.cuda_stream, N, T)
        except B.RnnError:
            empty_us = None
    r.close()

    peaks, peak_src = load_peaks()
    fl = phase_flops(cfg)
    if paths[0] == "wavefront":
        # the wavefront computes each step's input projection inside the
        # recurrent kernel; the input phase only packs the weights
        fl["rec_fwd"] += fl["input_gemm"]
        fl["input_gemm"] = 0.0
    total_flop = sum(fl.values())
    sm_clk = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    bf16_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])

    def phase_roof(ph):
        """(bound, peak TFLOP/s, note) of one phase, timed inside the step."""
        on_tensor = ph.endswith("gemm") or (ph == "rec_fwd" and paths[0] in ("tensor", "wavefront")) \
            or (ph == "rec_bwd" and paths[1] == "tensor")
        if on_tensor:
            if dt == "bf16":
                return "tensor", bf16_sus, "%s bf16 dense, sustained (cuBLAS loop)" % peak_src
            # every fp32 tensor-core phase (dense GEMMs and both recurrent
            # kernels) runs three kind::f16 passes on scaled fp16 hi / lo pairs
            return ("tensor", bf16_sus / 3.0,
                    "%s bf16 sustained / 3 passes: fp32 as three fp16 passes on "
                    "scaled hi / lo splits (fp16 and bf16 share the kind::f16 rate)"
                    % peak_src)
        return ("alu", fp32_simt_peak_tflops(num_sms, sm_clk),
                "fp32 FMA issue peak: %d SMs x 128 lanes x 2 flop x %.0f MHz (derived)"
                % (num_sms, sm_clk))

    per_phase = {}
    for ph in PHASE_NAMES:
        ms_ph = phases[ph][0] / max(1, args.steps)
        b_, pk_, _ = phase_roof(ph)
        ach = fl[ph] / (ms_ph * 1e-3) / 1e12 if ms_ph > 0 else 0.0
        per_phase[ph] = {"ms": round(ms_ph, 4), "kernels": phases[ph][1] / args.steps,
                         "algorithmic_tflop": round(fl[ph] / 1e12, 6), "bound": b_,
                         "achieved": round(ach, 3), "peak": round(pk_, 3),
                         "frac": round(ach / pk_, 4) if pk_ and fl[ph] else None}
        if ph in ("rec_fwd", "rec_bwd"):
            # serial steps of the phase: L * T layer steps, or T + L - 1
            # wavefront steps when all layers run in one launch
            wave = ph == "rec_fwd" and paths[0] == "wavefront"
            nsteps = (T + L - 1) if wave else L * T
            per_phase[ph]["path"] = paths[0] if ph == "rec_fwd" else paths[1]
            per_phase[ph]["us_per_step"] = round(ms_ph * 1e3 / nsteps, 3)
            if empty_us is not None and per_phase[ph]["path"] == "tensor" and L == 1:
                # latency bound of one serial step: max(W_hh streamed once
                # from on-chip memory at 128 B/clk/SM, the step's MMA work at
                # the phase's tensor peak) + the measured empty-step protocol
                G = gates(cfg["mode"])
                e = 2 if dt == "bf16" else 4
                w_us = G * H * H * e / (num_sms * 128.0 * sm_clk * 1e6) * 1e6
                mma_us = D * 2.0 * N * G * H * H / (pk_ * 1e12) * 1e6
                bound = max(w_us, mma_us) + empty_us
                per_phase[ph]["bound_us"] = {
                    "w_hh_stream_us": round(w_us, 3), "mma_us": round(mma_us, 3),
                    "empty_step_us": round(empty_us, 3), "bound_us": round(bound, 3),
                    "frac_of_bound": round(bound / per_phase[ph]["us_per_step"], 3),
                    "note": "empty step = the forward kernel's step protocol alone (exchange "
                            "words written and polled, one block barrier, partial-sum "
                            "pushes completing the owners' barriers; "
                            "rnn_measure_step_protocol), used for the backward too"}
    # dominant phase by time share
    dom = max(PHASE_NAMES, key=lambda p: phases[p][0])
    avg_ms = phases[dom][0] / max(1, args.steps)
    bound, peak, peak_note = phase_roof(dom)
    unit = "TFLOP/s"
    achieved = fl[dom] / (avg_ms * 1e-3) / 1e12 if avg_ms > 0 else 0.0
    value = aggregate_sequences_per_s(N, ws_n, ms_step_max)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "sequences/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if dt == "f32" else "bf16",
        "data": "synthetic (seeded N(0,1) inputs, U(-1/sqrt(H), 1/sqrt(H)) weights)",
        "config": {"workload": cfg["name"], "mode": cfg["mode"], "layers": L,
                   "bidirectional": cfg["bidir"], "T": T, "N": N, "I": I, "H": H,
                   "global_batch": N * ws_n, "seq_len": T,
                   "parallelism": ("dp%d (batch shards of %d sequences per GPU, dW/db "
                                   "all-reduce every step)" % (ws_n, N)) if ws_n > 1
                   else "single GPU",
                   "l2": "flushed before every timed step (256 MiB write, untimed)"},
        "effective_tflops": round(total_flop * ws_n / (ms_step_max * 1e-3) / 1e12, 3),
        "phases": per_phase,
        "recurrent_paths": {"fwd": paths[0], "bwd": paths[1]},
        "roofline": {"kernel": PHASE_KERNELS[dom], "phase": dom, "bound": bound,
                     "achieved": round(achieved, 3), "peak": round(peak, 3), "unit": unit,
                     "frac": round(achieved / peak, 4) if peak else None,
                     "traffic": traffic_for(dom, cfg), "peak_source": peak_note,
                     "algorithmic_flop_per_step": fl[dom],
                     "avg_phase_ms": round(avg_ms, 4)},
        "e2e": {"value": round(aggregate_sequences_per_s(N, ws_n, ms_e2e_max), 2), "unit": "sequences/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e_max, 4),
                "copies": "every step's inputs in from and results out to pinned host memory, "
                          "on two copy streams under the neighbouring steps' compute "
                          "(double-buffered on the device); the K steps timed as one region"},
        "varlen": {"value": round(aggregate_sequences_per_s(N, ws_n, ms_var_max), 2),
                   "unit": "sequences/s", "ms_per_step": round(ms_var_max, 4),
                   "recurrent_paths": {"fwd": vpaths[0], "bwd": vpaths[1]},
                   "lengths": "padded to T=%d; one sequence of length T, the others uniform "
                              "in [%d, %d] (mean %.1f); rnn_forward_training_varlen + "
                              "rnn_backward_data_varlen + rnn_backward_weights, L2 flushed "
                              "before every step"
                              % (T, (T + 1) // 2, T, float(lens_np.mean()))},
        "dropout": drop,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "wall_s_timed_region": round(wall, 3),
        "clocks": clocks,
    }
    return line


def run_reference(args, cfg):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    K, W = args.steps, args.warmup
    # the oracle, as it stands, on bounded samples; W warm-up + K timed samples
    budget = max(2.0, args.cpu_budget / max(1, K + W))
    vals = []
    sample = None
    for i in range(W + K):
        v, sample, _ = time_oracle(cfg, budget_s=budget, max_reps=1)
        if i >= W:
            vals.append(v)
    v = statistics.median(vals)
    line = {"metric": METRIC, "value": round(v, 4), "unit": "sequences/s", "n_gpus": ws_n,
            "steps": K, "warmup": W, "ms_per_step": round(cfg["N"] / v * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": cfg["name"], "T": cfg["T"], "N": cfg["N"], "I": cfg["I"],
                       "H": cfg["H"], "mode": cfg["mode"], "layers": cfg["L"],
                       "bidirectional": cfg["bidir"]},
            "cpu_baseline": {"value": round(v, 4), "unit": "sequences/s",
                             "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "sequences/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ds2_lstm", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gru", action="store_true",
                    help="time only the named workload (by default the ds2_lstm line also "
                         "carries the ds2_gru layer of the same shape)")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override T of the workload (small cases for profiler captures; "
                         "the default workload sizes are the benchmark)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    cfg = wl.WORKLOADS[args.workload]
    if args.seq_len > 0:
        cfg = wl.with_sizes(cfg, T=args.seq_len)
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
