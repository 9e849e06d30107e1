"""KDA forward benchmark on GB300: chunked prefill tokens/s (H=96, K=V=128) with
the decode steps/s beside it, each as a fraction of its HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0.  The headline ``value`` is whole-job prefill
throughput on the 4096-token, 96-head workload with inputs resident in HBM;
``e2e`` is the same metric through the public call with pinned host buffers
and the host<->device copies inside the timed region; ``decode`` is the
256-sequence single-token step repeated 64 times.  Each rank is an independent
replica (the sequences and heads of KDA are independent problems), so the job
processes N times the work and ``scaling`` is weak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KDA prefill tokens/s (H=96,K=V=128) + decode steps/s, % of roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def prefill_bytes(T_tokens: int, H: int, K: int, V: int, N: int, in_bytes: int, reads_state: bool) -> int:
    """Algorithmic HBM bytes of one chunked prefill: q, k, g [T,H,K] + v [T,H,V] + beta [T,H]
    read once, o [T,H,V] fp32 written once, final state [N,H,K,V] fp32 written once (and the
    initial state read once when given)."""
    per_token = H * ((3 * K + V) * in_bytes + in_bytes + V * 4)
    states = N * H * K * V * 4 * (2 if reads_state else 1)
    return T_tokens * per_token + states


# Bytes of one (64-token chunk, head) workspace slot of the tensor-core prefill
# (include/kda.h): what the chunk-local kernel writes and the state kernel reads.
SLOT_BYTES = 147968


def kernel_bytes(T_tokens: int, n_chunks: int, H: int, K: int, V: int, N: int, reads_state: bool, prologue: bool):
    """HBM bytes each kernel of the two-kernel prefill has to move by design:
    the chunk-local kernel reads q, k, v, g (bf16) and beta and writes one
    workspace slot per (chunk, head) (plus the prologue weights); the state
    kernel reads the slots and the initial state and writes o (fp32) and the
    final state."""
    local = T_tokens * H * ((3 * K + V) * 2 + 2) + n_chunks * H * SLOT_BYTES
    if prologue:  # conv weights, dt_bias and A_log, read once from HBM
        local += H * (2 * K + V) * 16 + H * K * 4 + K * 4
    state = n_chunks * H * SLOT_BYTES + T_tokens * H * V * 4 + N * H * K * V * 4 * (2 if reads_state else 1)
    return local, state


def decode_bytes(N: int, H: int, K: int, V: int, in_bytes: int) -> int:
    """One decode step: the fp32 state read and written once, plus q, k, g, v, beta and o."""
    return 2 * N * H * K * V * 4 + N * H * ((3 * K + V) * in_bytes + in_bytes + V * 4)


def source_sha(files) -> str:
    """Hash of the CUDA sources a kernel is built from (names relative to csrc/)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kimi_delta_attention_chunk_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(key: str):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json),
    if it was taken on the kernel's current sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(key)
    if not rec or rec.get("source_sha") != source_sha(rec.get("sources", [])):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [r for t, r in self.rows if self.t0 is None or (self.t0 - 0.1 <= t <= (self.t1 or t) + 0.1)]
        if not rows:
            rows = [r for _, r in self.rows]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle legs
def oracle_prefill_rate(H: int, T: int, heads: int, seed: int = 1):
    """Oracle tokens/s on `heads` of the H heads of a T-token prefill (scaled to all H)."""
    import oracle
    from kimi_delta_attention_chunk_gb300 import synth
    inp = synth.direct_inputs(T, heads, 128, 128, torch.bfloat16, seed=seed)
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=inp["scale"], nthreads=threads)
    dt = time.perf_counter() - t0
    return T * heads / H / dt, dt, threads


def cpu_baseline(H: int, T: int, budget_s: float = 12.0):
    """The oracle on the host cores: the whole T-token, H-head prefill, repeated
    until about budget_s seconds of work (at least once); mean tokens/s."""
    rates, total, reps, threads = [], 0.0, 0, 1
    while reps == 0 or total < budget_s:
        r, dt, threads = oracle_prefill_rate(H, T, H)
        rates.append(r)
        total += dt
        reps += 1
        if reps >= 50:
            break
    return {"value": sum(rates) / len(rates), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{reps} x ({T} tokens x {H} heads, K=V=128, bf16 inputs upcast to fp64), {total:.1f} s"}


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    H, T = 96, 4096
    heads = 4
    for _ in range(args.warmup):
        oracle_prefill_rate(H, T, heads)
    rates, total = [], 0.0
    for _ in range(args.steps):
        r, dt, threads = oracle_prefill_rate(H, T, heads)
        rates.append(r)
        total += dt
    value = sum(rates) / len(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "prefill B=1 T=4096 H=96 K=V=128 bf16 inputs, zero initial state",
                       "sample": f"{T} tokens x {heads} of {H} heads per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{T} tokens x {heads} of {H} heads per step, rate scaled to {H} heads"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU legs
def time_launches(fn, steps: int, stream):
    """Run fn() `steps` times; return (total ms, per-launch ms list) from CUDA events on `stream`."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), [a.elapsed_time(b) for a, b in ev]


def time_traced(kda, fn, steps: int, stream):
    """Like time_launches, with the prefill's own timing hook: per call the
    events before its first kernel, after the chunk-local kernel and after its
    last kernel.  Returns (total ms, per-call ms, chunk-local ms, state ms)."""
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    for trio in ev:
        for e in trio:
            e.record(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for b, sp, e in ev:
        kda.trace_events(b, sp, e)
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    per = [b.elapsed_time(e) for b, _, e in ev]
    k1 = [b.elapsed_time(sp) for b, sp, _ in ev]
    k2 = [sp.elapsed_time(e) for _, sp, e in ev]
    return t0.elapsed_time(t1), per, k1, k2


def sum_traffic(kernels):
    """DRAM bytes of one call (both kernels) from the committed ncu summary, or None."""
    t = [k["traffic"] for k in kernels]
    return None if any(x is None for x in t) else sum(t)


def kernel_split(k1, k2, local_bytes, state_bytes, hbm, traffic_keys):
    """Per-kernel live durations and design-traffic bandwidth of one call."""
    m1, m2 = sum(k1) / len(k1), sum(k2) / len(k2)
    out = []
    for name, ms, nbytes, key in (("chunk_local_kernel", m1, local_bytes, traffic_keys[0]),
                                   ("chunk_state_kernel", m2, state_bytes, traffic_keys[1])):
        gbs = nbytes / (ms * 1e-3) / 1e9
        out.append({"kernel": name, "ms": ms, "share": ms / (m1 + m2), "design_bytes": nbytes,
                    "design_gbs": gbs, "frac_of_hbm": gbs / hbm, "traffic": recorded_traffic(key)})
    return out


def run_ours(args, world, rank, local):
    import kimi_delta_attention_chunk_gb300 as kda
    from kimi_delta_attention_chunk_gb300 import synth

    kda.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    bf16_peak = float(peaks.get("bf16_tflops") or 1900.0)
    w = synth.WORKLOADS["prefill"]
    H, K, V, T = w.H, w.K, w.V, w.T
    host = synth.direct_inputs(T, H, K, V, w.dtype, w.seed + 1000 * rank)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    o = torch.empty((1, T, H, V), dtype=torch.float32, device=dev)
    sT = torch.empty((1, H, K, V), dtype=torch.float32, device=dev)
    # the caller-owned workspace and device status word, allocated once
    ws = torch.empty(kda.workspace_size(w.dtype, 1, T, H, K, V, 1, False), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def prefill():
        kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], o=o, final_state=sT,
                      workspace=ws, status=status)

    for _ in range(max(3, args.warmup)):
        prefill()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("t0")
    total_ms, per, k1, k2 = time_traced(kda, prefill, args.steps, stream)
    clocks.mark("t1")
    barrier(world)
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"prefill reported device status {int(status.item())}")
    total_ms = max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    tokens_per_step = T * world
    value = tokens_per_step / (ms_step * 1e-3)
    kernel_ms = sum(per) / len(per)
    pbytes = prefill_bytes(T, H, K, V, 1, 2, reads_state=False)
    achieved = pbytes / (kernel_ms * 1e-3) / 1e9
    lb, sb = kernel_bytes(T, (T + 63) // 64, H, K, V, 1, reads_state=False, prologue=False)
    kernels = kernel_split(k1, k2, lb, sb, hbm, ("chunk_local_kernel/prefill", "chunk_state_kernel/prefill"))

    # ---- end to end through the public call: pinned host in, host out.  Every step
    # uploads its inputs and downloads o and the final state; the steps are
    # pipelined over two device buffer sets, so the upload of step i+1 (one copy
    # stream) and the download of step i (another) overlap the prefill of step i.
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    names = ("q", "k", "v", "g", "beta")
    o_host = torch.empty_like(o, device="cpu").pin_memory()
    s_host = torch.empty_like(sT, device="cpu").pin_memory()
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in names)
    d2h = o_host.numel() * 4 + s_host.numel() * 4
    dbuf = [d, {k: (torch.empty_like(d[k]) if k in names else d[k]) for k in d}]
    obuf = [(o, sT), (torch.empty_like(o), torch.empty_like(sT))]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    step_i = [0]

    def e2e_step():
        b = step_i[0] % 2
        step_i[0] += 1
        x, (ox, sx) = dbuf[b], obuf[b]
        with torch.cuda.stream(s_up):
            s_up.wait_event(ev_done[b])  # step i-2 is done with these inputs
            for k in names:
                x[k].copy_(pin[k], non_blocking=True)
            ev_up[b].record(s_up)
        stream.wait_event(ev_up[b])
        stream.wait_event(ev_down[b])  # step i-2's outputs have left
        kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"], o=ox, final_state=sx,
                      workspace=ws)
        ev_done[b].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev_done[b])
            o_host.copy_(ox, non_blocking=True)
            s_host.copy_(sx, non_blocking=True)
            ev_down[b].record(s_down)

    def e2e_drain():
        stream.wait_stream(s_down)

    for _ in range(2):
        e2e_step()
    e2e_drain()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_up.wait_event(e0)
    for _ in range(args.steps):
        e2e_step()
    e2e_drain()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    e2e = {"value": tokens_per_step / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "pipelined": "upload, prefill and download of consecutive steps overlap"}
    del pin, o_host, s_host, dbuf, obuf

    # ---- decode: 256 sequences x 64 steps
    dw = synth.WORKLOADS["decode"]
    dec = synth.decode_inputs(dw.B, dw.H, dw.K, dw.V, dw.decode_steps, dw.dtype, dw.seed + 1000 * rank)
    dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in dec.items()}
    state = dd["state"].clone()
    od = torch.empty((dw.B, dw.H, dw.V), dtype=torch.float32, device=dev)
    steps = dw.decode_steps
    qs = [dd["q"][i] for i in range(steps)]
    ks = [dd["k"][i] for i in range(steps)]
    vs = [dd["v"][i] for i in range(steps)]
    gs = [dd["g"][i] for i in range(steps)]
    bs = [dd["beta"][i] for i in range(steps)]
    it = [0]

    def dstep():
        i = it[0] % steps
        it[0] += 1
        kda.recurrent_step(qs[i], ks[i], vs[i], gs[i], bs[i], state, scale=dd["scale"], o=od)

    for _ in range(max(3, args.warmup)):
        dstep()
    torch.cuda.synchronize()
    barrier(world)
    dsteps = steps * max(1, args.steps // 10)
    dec_ms, dper = time_launches(dstep, dsteps, stream)
    dec_ms = max_over_ranks(dec_ms, world) / dsteps
    dker = sum(dper) / len(dper)
    dbytes = decode_bytes(dw.B, dw.H, dw.K, dw.V, 2)
    dach = dbytes / (dker * 1e-3) / 1e9
    decode = {"value": world / (dec_ms * 1e-3), "unit": "steps/s", "tokens_per_s": world * dw.B / (dec_ms * 1e-3),
              "ms_per_step": dec_ms, "workload": "decode N=256 H=96 K=V=128 bf16, fp32 state in place, 64 steps",
              "roofline": {"bound": "hbm", "achieved": dach, "peak": hbm, "unit": "GB/s", "frac": dach / hbm,
                           "traffic": recorded_traffic("decode_step_kernel/decode"), "algorithmic_bytes": dbytes,
                           "peak_kind": peak_kind}}
    del dd, state, qs, ks, vs, gs, bs

    # ---- the layer's output gate on the prefill's o (4096 x 96 rows of 128):
    # reads o fp32 and the bf16 gate, writes fp32
    og_in = synth.output_gate_inputs((1, T, H, V), torch.bfloat16, 7 + 1000 * rank)
    og_o, og_g, og_w = (og_in[k].to(dev) for k in ("o", "gate", "weight"))
    og_out = torch.empty_like(og_o)

    def ogstep():
        kda.output_gate(og_o, og_g, og_w, out=og_out)

    for _ in range(max(3, args.warmup)):
        ogstep()
    torch.cuda.synchronize()
    barrier(world)
    og_ms, ogper = time_launches(ogstep, max(10, args.steps), stream)
    og_ms = max_over_ranks(og_ms, world) / max(10, args.steps)
    og_bytes = T * H * V * (4 + 2 + 4) + V * 4
    og_ach = og_bytes / (sum(ogper) / len(ogper) * 1e-3) / 1e9
    out_gate = {"value": world * T / (og_ms * 1e-3), "unit": "tokens/s", "ms_per_launch": og_ms,
                "workload": "output gate on the prefill's o: 4096 x 96 rows of 128, fp32 o, bf16 gate, fp32 out",
                "roofline": {"bound": "hbm", "achieved": og_ach, "peak": hbm, "unit": "GB/s", "frac": og_ach / hbm,
                             "traffic": recorded_traffic("output_gate_kernel/prefill"), "algorithmic_bytes": og_bytes, "peak_kind": peak_kind}}
    del og_in, og_o, og_g, og_w, og_out

    # ---- the projections ahead of the gate for the same 4096 tokens: x [4096, 7168]
    # -> gate_x [4096, 96*128] and beta [4096, 96] (rank-128 f_a/f_b, b_proj)
    GD, GR = 7168, 128
    gp_in = {k: v.to(dev) for k, v in synth.gate_proj_inputs(1, T, GD, GR, H * K, H, 9 + 1000 * rank).items()}
    gp_gx = torch.empty((1, T, H * K), dtype=torch.bfloat16, device=dev)
    gp_beta = torch.empty((1, T, H), dtype=torch.bfloat16, device=dev)
    gp_ws = torch.empty(kda.gate_proj_workspace_size(1, T, GD, GR, H), dtype=torch.uint8, device=dev)
    gp_status = torch.zeros(1, dtype=torch.int32, device=dev)

    def gpstep():
        kda.gate_proj(gp_in["x"], gp_in["f_a"], gp_in["f_b"], gp_in["b_proj"], gate_x=gp_gx, beta=gp_beta,
                      workspace=gp_ws, status=gp_status)

    for _ in range(max(3, args.warmup)):
        gpstep()
    torch.cuda.synchronize()
    barrier(world)
    gp_n = max(10, args.steps)
    gp_ms, gpper = time_launches(gpstep, gp_n, stream)
    if int(gp_status.item()) != 0:
        raise RuntimeError(f"gate projection reported device status {int(gp_status.item())}")
    gp_ms = max_over_ranks(gp_ms, world) / gp_n
    gp_bytes = 2 * (T * GD + GR * GD + H * GD + H * K * GR + T * H * K + T * H)
    gp_flops = 2 * T * (GD * (GR + H) + GR * H * K)
    gp_call = sum(gpper) / len(gpper)
    gp_ach = gp_bytes / (gp_call * 1e-3) / 1e9
    gate_proj = {"value": world * T / (gp_ms * 1e-3), "unit": "tokens/s", "ms_per_launch": gp_ms,
                 "workload": "gate projections for the prefill's 4096 tokens: x [4096, 7168] bf16, rank-128 "
                             "f_a/f_b to gate_x [4096, 96*128], b_proj + sigmoid to beta [4096, 96], bf16 out",
                 "gpu_launches": 3 * gp_n,
                 "tensor_tflops": gp_flops / (gp_call * 1e-3) / 1e12,
                 "roofline": {"bound": "hbm", "achieved": gp_ach, "peak": hbm, "unit": "GB/s", "frac": gp_ach / hbm,
                              "traffic": recorded_traffic("gate_proj/prefill"), "algorithmic_bytes": gp_bytes,
                              "peak_kind": peak_kind,
                              "note": "the three kernels of one call; algorithmic bytes exclude the round "
                                      "trips through the workspace (split partial sums and y)"}}
    del gp_in, gp_gx, gp_beta, gp_ws

    # ---- the backward of the 4096-token prefill (chunked, tensor cores); a
    # failure here is reported in its own line and does not stop the others
    dO = torch.randn((1, T, H, V), generator=torch.Generator(device=dev).manual_seed(11 + rank), device=dev)
    del ws
    bws = torch.empty(kda.bwd_workspace_size(w.dtype, 1, T, H, K, V, 1, False), dtype=torch.uint8, device=dev)

    def bwstep():
        kda.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO, scale=d["scale"], workspace=bws)

    bw_err = None
    try:
        bwstep()
        torch.cuda.synchronize()
    except Exception as exc:  # noqa: BLE001
        bw_err = str(exc)[:200]
    barrier(world)
    if max_over_ranks(0.0 if bw_err is None else 1.0, world) == 0.0:  # every rank ran it
        nb = 3
        bw_ms, bwper = time_launches(bwstep, nb, stream)
        bw_ms = max_over_ranks(bw_ms, world) / nb
        # algorithmic bytes: q, k, v, g (bf16), beta, dO (fp32) in; dq, dk, dv, dg, dbeta (fp32) out
        bw_bytes = T * H * ((3 * K + V) * 2 + 2 + 4 * V + (3 * K + V) * 4 + 4)
        bw_call = sum(bwper) / len(bwper)
        bw_gbs = bw_bytes / (bw_call * 1e-3) / 1e9
        # the method's multiply-adds of the backward's own products per (64-token chunk, head), one
        # term each (the hi|lo split runs three): the reverse chain's dU and dS, and the chunk kernel's
        # dO S^T, dU S^T, dO U^T, U dS'^T, [dBk | dBv], dM, and the gated back-products (U itself
        # comes from the forward's state kernel)
        chunks = (T + 63) // 64 * H
        bw_flops = 2 * chunks * (3670016 + 7864320)
        bw_tf = bw_flops / (bw_call * 1e-3) / 1e12
        backward = {"value": world * T / (bw_ms * 1e-3), "unit": "tokens/s", "ms_per_launch": bw_ms,
                    "workload": "backward of the 4096-token prefill (dq, dk, dv, dg, dbeta, dS0): the "
                                "tensor-core prefill again keeping every chunk's state, A and T, a reverse "
                                "tcgen05 chain carrying dS, chunk-parallel tcgen05 gradients",
                    "gpu_launches": 4 * nb,
                    "roofline": {"bound": "hbm", "achieved": bw_gbs, "peak": hbm, "unit": "GB/s",
                                 "frac": bw_gbs / hbm, "traffic": None, "algorithmic_bytes": bw_bytes,
                                 "tensor_tflops": bw_tf, "tensor_frac": bw_tf / bf16_peak,
                                 "algorithmic_flops": bw_flops,
                                 "note": "the chunk kernel dominates and is bound by the latency of its "
                                         "per-CTA scratch round trips, neither by HBM nor by the tensor pipe"}}
    else:
        backward = {"error": bw_err or "failed on another rank"}
    del dO, bws

    # ---- the other prefill workloads, each with its own roofline
    extra = {}
    for name in (["varlen"] if not args.skip_varlen else []) + (["long"] if not args.skip_long else []):
        wl = synth.WORKLOADS[name]
        inp = synth.device_inputs(name, dev, seed_offset=rank)
        Ttot = inp["beta"].shape[1]
        N = wl.n_seqs if wl.n_seqs else wl.B
        ox = torch.empty((1, Ttot, wl.H, wl.V), dtype=torch.float32, device=dev)
        sx = torch.empty((N, wl.H, wl.K, wl.V), dtype=torch.float32, device=dev)
        wsx = torch.empty(kda.workspace_size(wl.dtype, 1, Ttot, wl.H, wl.K, wl.V, N,
                                             inp.get("cu_seqlens") is not None), dtype=torch.uint8, device=dev)
        if wl.prologue:
            def run_x():
                kda.chunk_fwd_fused(inp["q_raw"], inp["k_raw"], inp["v_raw"], inp["gate_x"], inp["beta"],
                                    inp["conv_w"], inp["A_log"], inp["dt_bias"], scale=inp["scale"],
                                    initial_state=inp["initial_state"], o=ox, final_state=sx, workspace=wsx)
        else:
            def run_x():
                kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=inp["scale"],
                              initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"], o=ox, final_state=sx,
                              workspace=wsx)
        run_x()
        torch.cuda.synchronize()
        barrier(world)
        reps = 3
        xt, xper, xk1, xk2 = time_traced(kda, run_x, reps, stream)
        xt = max_over_ranks(xt, world) / reps
        xbytes = prefill_bytes(Ttot, wl.H, wl.K, wl.V, N, 2, reads_state=wl.init_state)
        xk = sum(xper) / len(xper)
        xach = xbytes / (xk * 1e-3) / 1e9
        if inp.get("cu_seqlens") is not None:
            cu = inp["cu_seqlens"].cpu().tolist()
            nch = sum((cu[i + 1] - cu[i] + 63) // 64 for i in range(len(cu) - 1))
        else:
            nch = (Ttot + 63) // 64
        xlb, xsb = kernel_bytes(Ttot, nch, wl.H, wl.K, wl.V, N, reads_state=wl.init_state, prologue=wl.prologue)
        xkernels = kernel_split(xk1, xk2, xlb, xsb, hbm,
                                (f"chunk_local_kernel/{name}", f"chunk_state_kernel/{name}"))
        extra[name] = {
            "value": world * Ttot / (xt * 1e-3), "unit": "tokens/s", "ms_per_launch": xt,
            "workload": ("varlen prefill: 16 sequences of 512..8192 tokens (%d total) packed by cu_seqlens, "
                         "H=96 K=V=128 bf16, fp32 initial states" % Ttot) if name == "varlen" else
                        ("long prefill with fused prologue (conv4, L2-norm, gate): T=65536 H=96 K=V=128 bf16, "
                         "nonzero initial state; prologue inside the chunk-local kernel"),
            "gpu_launches": reps * (3 if name == "varlen" else 2),
            "roofline": {"bound": "hbm", "achieved": xach, "peak": hbm, "unit": "GB/s", "frac": xach / hbm,
                         "traffic": sum_traffic(xkernels), "algorithmic_bytes": xbytes, "peak_kind": peak_kind,
                         "kernels": xkernels}}
        del inp, ox, sx, wsx

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill B=1 T=4096 H=96 K=V=128 bf16 inputs, fp32 state and output, "
                               "zero initial state", "parallelism": f"replicas x{world}",
                   "l2": "inputs (611 MB per step) larger than L2; no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": sum_traffic(kernels), "algorithmic_bytes": pbytes,
                     "kernel_ms": kernel_ms, "peak_kind": peak_kind, "kernels": kernels},
        "clocks": clk, "e2e": e2e, "gpu_launches": 2 * args.steps,
        "decode": decode,
        "output_gate": out_gate,
        "gate_proj": gate_proj,
        "backward": backward,
    }
    line.update(extra)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(H, T)
    print(json.dumps(line), flush=True)


def profile_case(args):
    """A few launches of one kernel on a chosen size, for ncu captures (prints 'ok')."""
    import kimi_delta_attention_chunk_gb300 as kda
    from kimi_delta_attention_chunk_gb300 import synth
    dev = torch.device("cuda", 0)
    if args.profile_case == "prefill":
        inp = synth.direct_inputs(args.profile_T, args.profile_H, 128, 128, torch.bfloat16, seed=1)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        for _ in range(args.profile_reps):
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"])
    elif args.profile_case == "fused":
        inp = synth.prologue_inputs(args.profile_T, args.profile_H, 128, 128, torch.bfloat16, seed=4)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        for _ in range(args.profile_reps):
            kda.chunk_fwd_fused(d["q_raw"], d["k_raw"], d["v_raw"], d["gate_x"], d["beta"], d["conv_w"],
                                d["A_log"], d["dt_bias"], scale=d["scale"], initial_state=d["initial_state"])
    elif args.profile_case == "gate_proj":
        gp = {k: v.to(dev) for k, v in synth.gate_proj_inputs(1, args.profile_T, 7168, 128, args.profile_H * 128,
                                                               args.profile_H, 9).items()}
        for _ in range(args.profile_reps):
            kda.gate_proj(gp["x"], gp["f_a"], gp["f_b"], gp["b_proj"])
    elif args.profile_case == "bwd":
        d = synth.device_inputs("prefill", dev)
        if args.profile_bwd_H < d["q"].shape[2]:  # the first heads of the 4096-token workload
            d = {k: (v[:, :, :args.profile_bwd_H].contiguous() if k in ("q", "k", "v", "g", "beta") else v)
                 for k, v in d.items()}
        dO = torch.randn(d["q"].shape[:3] + (d["v"].shape[-1],), device=dev,
                         generator=torch.Generator(device=dev).manual_seed(11))
        for _ in range(args.profile_reps):
            kda.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO, scale=d["scale"])
    elif args.profile_case == "output_gate":
        og = synth.output_gate_inputs((1, args.profile_T, args.profile_H, 128), torch.bfloat16, 7)
        o, g, wt = (og[k].to(dev) for k in ("o", "gate", "weight"))
        out = torch.empty_like(o)
        for _ in range(args.profile_reps):
            kda.output_gate(o, g, wt, out=out)
    else:
        w = synth.WORKLOADS["decode"]
        dec = synth.decode_inputs(w.B, w.H, w.K, w.V, args.profile_reps, w.dtype, w.seed)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in dec.items()}
        state = d["state"].clone()
        for i in range(args.profile_reps):
            kda.recurrent_step(d["q"][i], d["k"][i], d["v"][i], d["g"][i], d["beta"][i], state, scale=d["scale"])
    torch.cuda.synchronize()
    print("ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile-case", choices=["prefill", "fused", "decode", "output_gate", "gate_proj", "bwd"], default=None,
                    help="run a few launches of one kernel for an ncu capture instead of the benchmark")
    ap.add_argument("--profile-T", type=int, default=2048)
    ap.add_argument("--profile-H", type=int, default=16)
    ap.add_argument("--profile-reps", type=int, default=2)
    ap.add_argument("--profile-bwd-H", type=int, default=96,
                    help="bwd case: heads of the 4096-token workload to run (default all 96)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-varlen", action="store_true", help="skip the 16-sequence varlen prefill line")
    ap.add_argument("--skip-long", action="store_true", help="skip the 65536-token fused-prologue line")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args)
        return
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
