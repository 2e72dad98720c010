"""Benchmark: forward tokens/s and fraction of the GB300 roofline for the
chunkwise gated delta rule, gated DeltaNet at B=4, H=16, T=2048, d=128, bf16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one dn_chunk_fwd call over the whole workload (all chunk steps of
the path in one launch).  Inputs are resident in HBM before the timed region;
L2 is flushed before every timed step, outside the events
that time the step.  Each rank runs its own copy of the workload (independent
sequences, no exchange between GPUs), so scaling is weak and `value` is the
tokens all ranks processed per second of the slowest rank.

`--impl reference` times the fp64 CPU oracle on the host cores instead (on a
bounded sample of the same workload per step); under torchrun only rank 0
runs it.  One JSON line is printed by rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "fwd tokens/s & % of roofline, gated delta rule H=16 d=128 T=2048 (1 GB300)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
E2E_NOTE = ("every step copies its inputs from pinned host memory to the device, makes the call "
            "and copies the results back to pinned host memory; the inputs sit in one pinned "
            "staging buffer and the results in one device buffer (each tensor at a 256-byte "
            "aligned offset), so each direction is one copy per step; steps run as a three-stage "
            "pipeline (copy-in stream, compute stream, copy-out stream; double-buffered), timed "
            "from the first copy in to the last copy out")
# The same string in both arms' config, so that the two lines name one
# workload and one timing rule (the reference arm runs on host cores).
L2_NOTE = ("GPU arm: L2 flushed before every timed step, outside the step's events: a 256 MiB "
           "write, then a 256 MiB read of another buffer so the written lines are back in HBM "
           "and L2 holds only clean unrelated lines; reference arm: host cores, no device cache")


class L2Flush:
    """Before each timed step: write a buffer larger than L2, then read another
    one, so that neither the step's inputs nor dirty lines of the flush itself
    are in L2 when the step starts."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = os.path.join(ROOT, "chunkwise_gated_delta_chunk_gb300", "csrc")


# --------------------------------------------------------------------------
# Algorithmic work of one forward (full C x C tiles; solve and elementwise
# terms excluded), per token and per state.
# --------------------------------------------------------------------------
def algorithmic(inp: dict) -> dict:
    B, T, Nk, dk = inp["q"].shape
    Nv, dv = inp["v"].shape[2], inp["v"].shape[3]
    C = 64
    tok = B * T
    e = inp["q"].element_size()
    has_g = inp["g"] is not None
    has_h0 = inp["h0"] is not None
    has_ht = True
    N = inp["N"]
    flops = tok * (Nv * (6 * dk * dv + 2 * C * (dk + 2 * dv)) + Nk * (4 * C * dk))
    bytes_ = (tok * (2 * Nk * dk * e + 2 * Nv * dv * e + Nv * 4 * (1 + has_g))
              + N * Nv * dk * dv * 4 * (has_h0 + has_ht))
    return dict(flops=flops, bytes=bytes_, tokens=tok)


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm_gbs=float(pk["hbm_gbs"]), bf16_tflops=float(pk["bf16_tflops"]),
                    bf16_tflops_sustained=float(pk.get("bf16_tflops_sustained",
                                                       pk["bf16_tflops"]))), "measured"
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0), "fallback"


def sources_hash() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(KERNEL_SOURCES)):
        with open(os.path.join(KERNEL_SOURCES, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload, {}).get(kernel)
    if not ent or ent.get("sources") != sources_hash():
        return None
    return ent.get("bytes_per_launch")


# --------------------------------------------------------------------------
# Clock sampling during the timed region.
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.gpu_id = gpu_id

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the first sample land before the timed region
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in load),
                    sm_max_mhz=max(r["smax"] for r in rows), reasons=sorted(reasons),
                    samples=len(rows), samples_under_load=len(load),
                    power_w_max=max(r["power"] for r in rows))


def smi_gpu_id(dev, local: int) -> str:
    """nvidia-smi id (UUID) of the CUDA device, matched by UUID."""
    try:
        want = str(torch.cuda.get_device_properties(dev).uuid).lower().replace("gpu-", "")
        out = subprocess.run(["nvidia-smi", "--query-gpu=uuid", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=30).stdout
        for line in out.splitlines():
            u = line.strip()
            if u.lower().replace("gpu-", "") == want:
                return u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis:
        return vis.split(",")[local].strip()
    return str(local)


# --------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm).
# --------------------------------------------------------------------------
def oracle_time(inp: dict, units, threads: int = 0) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["h0"],
                     inp["cu_seqlens"], inp["scale"], units=units, threads=threads,
                     use_qk_l2norm_in_kernel=inp.get("qk_l2norm", False))
    return time.perf_counter() - t0


def oracle_sample(inp: dict, budget_s: float):
    """Units of the workload whose oracle run takes about `budget_s` seconds
    on all host cores.  Returns (units, tokens, seconds, cores)."""
    import oracle
    cores = oracle.default_threads()
    Nv = inp["v"].shape[2]
    n_units = inp["N"] * Nv
    per_unit_tokens = workloads.tokens(inp) / max(inp["N"], 1)
    # one unit on one core to size the sample
    t1 = oracle_time(inp, [0], threads=1)
    want = max(1, min(n_units, int(budget_s * cores / max(t1, 1e-6))))
    # whole waves of `cores` units keep every core busy
    if want >= cores:
        want = (want // cores) * cores
    units = list(range(want))
    return units, int(per_unit_tokens * want / Nv), cores


def reference_arm(args, inp, wl_name, rank, world):
    if rank != 0:
        return
    import oracle
    cores = oracle.default_threads()
    steps, warm = args.steps, args.warmup
    # size each step so that (warmup + steps) finishes in about two minutes
    t1 = oracle_time(inp, [0], threads=1)
    Nv = inp["v"].shape[2]
    budget = 120.0 / max(steps + warm, 1)
    n_units = max(1, min(inp["N"] * Nv, int(budget * cores / max(t1, 1e-6))))
    units = list(range(n_units))
    tok_step = workloads.tokens(inp) * n_units / (inp["N"] * Nv)
    for _ in range(warm):
        oracle_time(inp, units)
    times = [oracle_time(inp, units) for _ in range(steps)]
    sec = sum(times)
    value = tok_step * steps / sec
    sample = "%d of %d (sequence, v-head) units per step (%.0f token-heads of %d)" % (
        n_units, inp["N"] * Nv, tok_step * Nv, workloads.tokens(inp) * Nv)
    line = dict(metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=steps, warmup=warm,
                ms_per_step=1e3 * sec / steps, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic", impl="reference",
                config=dict(config_of(wl_name, inp, chunk=args.chunk, l2=L2_NOTE), mode=args.mode),
                cpu_baseline=dict(value=value, unit=UNIT, cores=cores, kind="oracle",
                                  sample=sample),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def packed(like: dict, device=None, pin=False):
    """One byte buffer holding a tensor of each shape and dtype in `like`
    (256-byte aligned offsets) and the tensor views into it."""
    offs, total = {}, 0
    for key, val in like.items():
        offs[key] = total
        total += (val.numel() * val.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = {}
    for key, val in like.items():
        n = val.numel() * val.element_size()
        views[key] = buf[offs[key]:offs[key] + n].view(val.dtype).view(val.shape)
    return buf, views


def pipelined_e2e(dev, stream, host: dict, dev_outputs, launch, E: int, warm: int = 3):
    """Milliseconds per step of the end-to-end loop through the public API.

    Every step copies its inputs from pinned host memory to the device, makes
    the call, and copies its results back to pinned host memory.  The steps
    run as a three-stage pipeline: the copies in on their own stream, the
    call on the compute stream `stream`, the copies out on a third stream;
    inputs and results are double-buffered on the device (and the results
    on the host).  (Spreading the copies over more streams measured no
    faster: the host-to-device link, not one copy engine, is the limit.)
    So step i's copies overlap the calls of steps i - 1 and i + 1, as in a
    serving loop.  The inputs sit in one pinned staging buffer and each
    step's results in one device buffer (`packed`), so that each direction
    is a single copy per step (one copy per tensor measured ≈ 8 % slower:
    the six input copies each pay a fixed cost).  `dev_outputs()` makes one
    set of device result tensors (a dict, for their shapes and dtypes);
    `launch(inputs, outputs)` enqueues the call on `stream`.  Returns the
    milliseconds per step, timed from the first copy in to the last copy
    out, and the bytes each step copies in and out."""
    NB, NIN, NOUT = 2, 1, 1  # buffers; copy-in and copy-out streams
    s_in = [torch.cuda.Stream(dev) for _ in range(NIN)]
    s_out = [torch.cuda.Stream(dev) for _ in range(NOUT)]
    hin_raw, hin = packed(host, pin=True)
    for key, val in host.items():
        hin[key].copy_(val)
    dbuf = [packed(host, device=dev) for _ in range(NB)]
    like_out = dev_outputs()
    outs = [packed(like_out, device=dev) for _ in range(NB)]
    hout = [packed(like_out, pin=True)[0] for _ in range(NB)]
    ev_in = [[torch.cuda.Event() for _ in range(NIN)] for _ in range(NB)]
    ev_comp = [torch.cuda.Event() for _ in range(NB)]
    ev_out = [[torch.cuda.Event() for _ in range(NOUT)] for _ in range(NB)]
    for b in range(NB):
        ev_comp[b].record(stream)
        for e in ev_out[b]:
            e.record(stream)

    def step(i):
        b = i % NB
        for j, st in enumerate(s_in):
            st.wait_event(ev_comp[b])  # the call that read buffer b is done
            with torch.cuda.stream(st):
                dbuf[b][0].copy_(hin_raw, non_blocking=True)
            ev_in[b][j].record(st)
        for e in ev_in[b]:
            stream.wait_event(e)
        for e in ev_out[b]:
            stream.wait_event(e)  # results of buffer b are on the host
        launch(dbuf[b][1], outs[b][1])
        ev_comp[b].record(stream)
        for j, st in enumerate(s_out):
            st.wait_event(ev_comp[b])
            with torch.cuda.stream(st):
                hout[b].copy_(outs[b][0], non_blocking=True)
            ev_out[b][j].record(st)

    for i in range(warm):
        step(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in[0])
    for st in s_in[1:]:
        st.wait_event(e0)
    for i in range(E):
        step(warm + i)
    for st in s_out[1:]:
        done = torch.cuda.Event()
        done.record(st)
        s_out[0].wait_event(done)
    e1.record(s_out[0])
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / E, hin_raw.numel(), outs[0][0].numel()


def launches_per_call(kernel: str) -> int:
    """Kernels one call launches: dn_last_kernel() lists them joined by '+'."""
    return len([k for k in kernel.split("+") if k])


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest value of `x` over all ranks (the slowest rank's time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Tokens all ranks processed per second of the slowest rank."""
    return tokens_per_rank * world / (ms_max / 1e3)


def config_of(wl_name, inp, l2, chunk=64):
    B, T, Nk, dk = inp["q"].shape
    Nv, dv = inp["v"].shape[2], inp["v"].shape[3]
    return dict(workload=wl_name, B=B, T=T, Nk=Nk, Nv=Nv, dk=dk, dv=dv, chunk=chunk,
                global_batch=B, seq_len=T, gate=inp["g"] is not None,
                h0=inp["h0"] is not None, qk_l2norm_in_kernel=bool(inp.get("qk_l2norm")), l2=l2)


# --------------------------------------------------------------------------
# Backward (dn_chunk_bwd): same timing rules, its own algorithmic work.
# --------------------------------------------------------------------------
BWD_METRIC = "bwd tokens/s & % of roofline, gated delta rule H=16 d=128 T=2048 (1 GB300)"


def algorithmic_bwd(inp: dict) -> dict:
    """Work of one backward: the forward it reruns plus the products of the
    chunk-form gradient (per chunk and value head: eight C x dk x dv products,
    five C x C x dv, four C x C x dk; per key head K K^T and Q K^T again).
    Bytes: q, k, v, dO, beta, g in; dq, dk, dv (fp32), dbeta, dg out; h0,
    dht in and dh0 out."""
    B, T, Nk, dk = inp["q"].shape
    Nv, dv = inp["v"].shape[2], inp["v"].shape[3]
    C = 64
    tok = B * T
    e = inp["q"].element_size()
    has_g = inp["g"] is not None
    has_h0 = inp["h0"] is not None
    N = inp["N"]
    fwd = algorithmic(inp)
    flops = fwd["flops"] + tok * (Nv * (16 * dk * dv + 10 * C * dv + 8 * C * dk) + Nk * 4 * C * dk)
    bytes_ = (tok * (2 * Nk * dk * e + 2 * Nv * dv * e + Nv * 4 * (1 + has_g)
                     + 4 * (2 * Nk * dk + Nv * dv) + Nv * 4 * (1 + has_g))
              + N * Nv * dk * dv * 4 * (2 * has_h0 + 1))
    return dict(flops=flops, bytes=bytes_, tokens=tok)


def fp32_alu_peak_tflops(sm_mhz: float) -> float:
    """fp32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 flop x clock."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


def bench_bwd(args, inp, wl_name, dn, dev, rank, world, dist):
    d = workloads.to_device(inp, dev)
    B, T, Nk, dk = d["q"].shape
    Nv, dv = d["v"].shape[2], d["v"].shape[3]
    N = inp["N"]
    gen = torch.Generator().manual_seed(1234)
    inp = dict(inp)
    inp["do"] = torch.randn(inp["v"].shape, generator=gen).to(inp["v"].dtype)
    inp["dht"] = torch.randn(N, Nv, dk, dv, generator=gen)
    d["do"], d["dht"] = inp["do"].to(dev), inp["dht"].to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    grads = dict(dq=torch.empty(d["q"].shape, **f32), dk=torch.empty(d["k"].shape, **f32),
                 dv=torch.empty(d["v"].shape, **f32), dbeta=torch.empty(d["beta"].shape, **f32),
                 dg=None if d["g"] is None else torch.empty(d["beta"].shape, **f32),
                 dh0=None if d["h0"] is None else torch.empty(N, Nv, dk, dv, **f32))
    dt = dn.dtype_code(d["q"].dtype)
    ws = torch.empty(max(dn.dn_chunk_bwd_workspace_bytes(N, B, T, Nk, Nv, dk, dv, dt), 16),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def launch(src=d):
        st = dn.dn_chunk_bwd(src["q"], src["k"], src["v"], src["beta"], src["g"], src["h0"],
                             src["cu_seqlens"], N, B, T, Nk, Nv, dk, dv, dt, inp["scale"], 0,
                             src["do"], src["dht"], grads["dq"], grads["dk"], grads["dv"],
                             grads["dbeta"], grads["dg"], grads["dh0"], ws, stream=stream)
        if st != dn.DN_OK:
            raise dn.DnError(st, "dn_chunk_bwd")

    flush = L2Flush(dev)
    for _ in range(args.warmup):
        flush()
        launch()
    torch.cuda.synchronize(dev)
    if dn.dn_check(stream) != dn.DN_OK:
        raise RuntimeError("warm-up reported a device error")
    kernel = dn.dn_last_kernel()
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(smi_gpu_id(dev, int(os.environ.get("LOCAL_RANK", "0")))) as clk:
        for i in range(K):
            flush()
            ev0[i].record(stream)
            launch()
            ev1[i].record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    ms = sum(a.elapsed_time(b) for a, b in zip(ev0, ev1)) / K
    if dn.dn_check(stream) != dn.DN_OK:
        raise RuntimeError("timed region reported a device error")
    ms_max = max_over_ranks(ms, dist, dev)

    # end to end: inputs and output gradient from pinned host memory, every
    # gradient back to the host, pipelined over three streams
    host = {key: inp[key].contiguous().pin_memory() for key in
            ("q", "k", "v", "beta", "g", "h0", "cu_seqlens", "do", "dht") if inp[key] is not None}

    def e2e_launch(src, dst):
        st = dn.dn_chunk_bwd(src["q"], src["k"], src["v"], src["beta"], src.get("g"), src.get("h0"),
                             src.get("cu_seqlens"), N, B, T, Nk, Nv, dk, dv, dt, inp["scale"], 0,
                             src["do"], src["dht"], dst["dq"], dst["dk"], dst["dv"], dst["dbeta"],
                             dst.get("dg"), dst.get("dh0"), ws, stream=stream)
        if st != dn.DN_OK:
            raise dn.DnError(st, "dn_chunk_bwd")

    # (h2d, d2h: the bytes each step copies, staging alignment included)
    e2e_ms, h2d, d2h = pipelined_e2e(dev, stream, host,
                                     lambda: {key: torch.empty_like(val) for key, val in grads.items()
                                              if val is not None},
                                     e2e_launch, max(1, min(args.e2e_steps, 10)), warm=2)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    alg = algorithmic_bwd(inp)
    clocks = clk.summary()
    sec = ms / 1e3
    mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
    achieved = alg["flops"] / sec / 1e12
    peaks, peak_src = load_peaks()
    alu = fp32_alu_peak_tflops(mhz)
    if "tf32" in kernel:
        # the reverse walk's products run as TF32 tensor-core tiles: TF32 dense
        # peak = the bf16 GEMM peak x the nominal TF32 / bf16 ratio (1.1 / 2.25)
        peak = peaks["bf16_tflops"] * 1.1 / 2.25
        bound, src = "tensor", ("%s bf16 %.0f TFLOP/s x 1.1 / 2.25 (nominal TF32 / bf16)"
                                % (peak_src, peaks["bf16_tflops"]))
    else:
        peak = alu
        bound, src = "alu", "derived: 152 SMs x 128 fp32 lanes x 2 flop x %.0f MHz" % mhz
    roof = dict(bound=bound, achieved=achieved, peak=peak, unit="TFLOP/s", frac=achieved / peak,
                traffic=measured_traffic(kernel, wl_name + ":bwd"),
                peak_source=src, fp32_alu_peak=alu, frac_of_fp32_alu=achieved / alu,
                roofline_time_us=1e6 * max(alg["flops"] / (peak * 1e12),
                                           alg["bytes"] / (peaks["hbm_gbs"] * 1e9)),
                algorithmic_bytes=alg["bytes"], algorithmic_flops=alg["flops"],
                hbm_gbs=alg["bytes"] / sec / 1e9, kernel=kernel)
    line = dict(metric=BWD_METRIC, value=weak_scaling_value(alg["tokens"], world, ms_max), unit=UNIT,
                n_gpus=world, steps=K, warmup=args.warmup, ms_per_step=ms_max,
                higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype=("tf32 (fp32 accumulation; inputs bf16)" if "tf32" in kernel
                       else "f32 (inputs %s)" % ("bf16" if d["q"].dtype == torch.bfloat16 else "f32")),
                data="synthetic",
                config=dict(config_of(wl_name, inp, l2=L2_NOTE), mode="bwd"),
                parallelism="dp%d (independent sequences per GPU, no collective)" % world,
                gpu_launches=K * launches_per_call(kernel), roofline=roof,
                e2e=dict(value=weak_scaling_value(alg["tokens"], world, e2e_ms), unit=UNIT,
                         h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h, ms_per_step=e2e_ms,
                         schedule=E2E_NOTE),
                clocks=clocks)
    if not args.no_cpu_baseline and world == 1:
        import oracle
        cores = oracle.default_threads()
        groups = list(range(min(N * Nk, cores)))
        t0 = time.perf_counter()
        oracle.recurrent_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["h0"],
                             inp["cu_seqlens"], inp["scale"], do=inp["do"], dht=inp["dht"],
                             groups=groups)
        secs = time.perf_counter() - t0
        toks = workloads.tokens(inp) * len(groups) / (N * Nk)
        line["cpu_baseline"] = dict(
            value=toks / secs, unit=UNIT, cores=cores, kind="oracle",
            sample="%d of %d (sequence, key head) groups of the workload, one pass (%.1f s)" % (
                len(groups), N * Nk, secs))
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=workloads.HEADLINE, choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--chunk", type=int, default=64, choices=[16, 32, 64],
                    help="chunk length C (16 and 32 run the CUDA-core kernel)")
    ap.add_argument("--mode", default="chunk", choices=["chunk", "recurrent", "bwd"],
                    help="dn_chunk_fwd (default), the token-serial dn_recurrent_fwd, or the "
                         "backward dn_chunk_bwd")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)

    wl_name = args.workload
    inp = workloads.workload_inputs(wl_name)

    if args.impl == "reference":
        reference_arm(args, inp, wl_name, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return

    import chunkwise_gated_delta_chunk_gb300 as dn
    dn.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.mode == "bwd":
        bench_bwd(args, inp, wl_name, dn, dev, rank, world, dist)
        return
    d = workloads.to_device(inp, dev)
    B, T, Nk, dk = d["q"].shape
    Nv, dv = d["v"].shape[2], d["v"].shape[3]
    N = inp["N"]
    o = torch.empty(B, T, Nv, dv, dtype=d["q"].dtype, device=dev)
    ht = torch.empty(N, Nv, dk, dv, dtype=torch.float32, device=dev)
    dt = dn.dtype_code(d["q"].dtype)
    stream = torch.cuda.current_stream(dev)

    ws = dn.workspace_for(d["q"], d["v"], N, args.chunk)
    flags = dn.DN_QK_L2NORM if inp.get("qk_l2norm") else 0

    def launch(q=d["q"], k=d["k"], v=d["v"], beta=d["beta"], g=d["g"], h0=d["h0"],
               cu=d["cu_seqlens"], o=o, ht=ht):
        if args.mode == "recurrent":
            st = dn.dn_recurrent_fwd(q, k, v, beta, g, h0, cu, N, B, T, Nk, Nv, dk, dv, dt,
                                     inp["scale"], o, ht, stream=stream, flags=flags)
        else:
            st = dn.dn_chunk_fwd(q, k, v, beta, g, h0, cu, N, B, T, Nk, Nv, dk, dv, dt,
                                 inp["scale"], args.chunk, o, ht, ws, stream=stream, flags=flags)
        if st != dn.DN_OK:
            raise dn.DnError(st)

    flush = L2Flush(dev)
    for _ in range(args.warmup):
        flush()
        launch()
    torch.cuda.synchronize(dev)
    st = dn.dn_check(stream)
    if st != dn.DN_OK:
        raise dn.DnError(st, "warm-up")
    kernel = dn.dn_last_kernel()

    # ---------------- device-timed region --------------------------------
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    gpu_id = smi_gpu_id(dev, local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_id) as clk:
        w0 = time.perf_counter()
        for i in range(K):
            flush()
            ev0[i].record(stream)
            launch()
            ev1[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - w0
    if dist is not None:
        dist.barrier()
    per = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    ms = sum(per) / K
    st = dn.dn_check(stream)
    if st != dn.DN_OK:
        raise dn.DnError(st, "timed region")
    ms_max = max_over_ranks(ms, dist, dev)

    # ---------------- end to end through the public API -------------------
    # per step: pinned host -> device copies of the inputs, the call, and the
    # device -> host read of o and ht, pipelined over three streams
    host = {}
    for key in ("q", "k", "v", "beta", "g", "h0", "cu_seqlens"):
        if inp[key] is not None:
            host[key] = inp[key].contiguous().pin_memory()

    def e2e_launch(src, dst):
        launch(q=src["q"], k=src["k"], v=src["v"], beta=src["beta"], g=src.get("g"),
               h0=src.get("h0"), cu=src.get("cu_seqlens"), o=dst["o"], ht=dst["ht"])

    # (h2d, d2h: the bytes each step copies, staging alignment included)
    e2e_ms, h2d, d2h = pipelined_e2e(dev, stream, host,
                                     lambda: dict(o=torch.empty_like(o), ht=torch.empty_like(ht)),
                                     e2e_launch, args.e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)

    if rank != 0:
        dist.destroy_process_group()
        return

    # ---------------- roofline --------------------------------------------
    alg = algorithmic(inp)
    peaks, peak_src = load_peaks()
    sec = ms / 1e3
    achieved_gbs = alg["bytes"] / sec / 1e9
    tflops = alg["flops"] / sec / 1e12
    t_hbm = alg["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg["flops"] / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    if bound == "hbm":
        roof = dict(bound="hbm", achieved=achieved_gbs, peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=achieved_gbs / peaks["hbm_gbs"])
    else:
        roof = dict(bound="tensor", achieved=tflops, peak=peaks["bf16_tflops"],
                    unit="TFLOP/s", frac=tflops / peaks["bf16_tflops"])
    roof["traffic"] = measured_traffic(kernel, wl_name)
    roof["peak_source"] = peak_src
    roof["roofline_time_us"] = 1e6 * max(t_hbm, t_tc)
    roof["algorithmic_bytes"] = alg["bytes"]
    roof["algorithmic_flops"] = alg["flops"]
    roof["tflops"] = tflops
    roof["kernel"] = kernel

    line = dict(metric=METRIC, value=weak_scaling_value(alg["tokens"], world, ms_max), unit=UNIT,
                n_gpus=world, steps=K, warmup=args.warmup, ms_per_step=ms_max,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16"
                if d["q"].dtype == torch.bfloat16 else "f32", data="synthetic",
                config=dict(config_of(wl_name, inp, chunk=args.chunk, l2=L2_NOTE), mode=args.mode),
                parallelism="dp%d (independent sequences per GPU, no collective)" % world,
                gpu_launches=K * launches_per_call(kernel), roofline=roof,
                e2e=dict(value=weak_scaling_value(alg["tokens"], world, e2e_ms), unit=UNIT,
                         h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                         ms_per_step=e2e_ms, schedule=E2E_NOTE),
                wall_ms_timed_loop=1e3 * wall)
    clocks = clk.summary()
    line["clocks"] = clocks
    if not args.no_cpu_baseline and world == 1:
        units, toks, cores = oracle_sample(inp, budget_s=15.0)
        secs = oracle_time(inp, units)
        line["cpu_baseline"] = dict(
            value=toks / secs, unit=UNIT, cores=cores, kind="oracle",
            sample="%d of %d (sequence, v-head) units of the workload, one pass (%.1f s)" % (
                len(units), inp["N"] * Nv, secs))
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
