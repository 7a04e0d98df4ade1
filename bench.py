#!/usr/bin/env python
"""Benchmark of the GMA forward pass on GB300: tokens/s and fraction of roofline.

One step = one full forward pass (responsibilities of queries and keys, write phase, read
phase) over the workload's synthetic inputs, which are resident in HBM before timing starts.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gma|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own independent
replica on its own heads (the (batch, head) slices do not interact), so per-GPU work is fixed
and ``scaling`` is "weak"; the only collectives are the timing barrier and the max over ranks.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same workload (the
only reference this method has: the page publishes no implementation).
"""
import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_latent_routing_gb300 import inputs as W  # noqa: E402

METRIC = "GMA causal fwd tokens/s at N=65536,K=128 on 1 GB300; % of roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = W.LONG_CAUSAL.name
L2_BYTES = 129 * 2 ** 20
SMS = 152
FP32_LANES_PER_SM = 128


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


# ----------------------------------------------------------------------------- work model
def path_bytes(w):
    """Algorithmic bytes of one step: Q_X, K_X, V read once and O written once."""
    esz = 2 if w.dtype == "bf16" else 4
    return (w.token_heads + w.key_heads) * esz * (w.d_r + w.d_v)


def path_flops(w):
    """Algorithmic flops of one step: the two [x^2, x] contractions (8 d_r K) plus the write and
    read contractions including the normaliser (4 K (d_v + 1)), per token-head."""
    return (w.token_heads + w.key_heads) * (4 * w.d_r * w.K + 2 * w.K * (w.d_v + 1))


def kernel_work(w, name):
    """(bound, amount, unit) of one launch of the named kernel.  Tensor-core kernels count
    algorithmic bytes or flops of the steps they fuse; CUDA-core kernels count their fp32
    arithmetic (bound "alu")."""
    th = w.token_heads
    esz = 2 if w.dtype == "bf16" else 4
    if name == "tc_causal_chunked":
        # the output pass reads Q_X and V and writes O (K_X is read by the segment pass; the
        # stored Gamma_K it also reads is not algorithmic traffic)
        return "hbm", th * esz * (w.d_r + 2 * w.d_v), "GB/s"
    if name == "tc_causal_single_launch":
        # the whole causal path in one launch: Q_X, K_X and V read once, O written (its second
        # sweep's re-read of K_X and V, and the segment memories it exchanges, are not
        # algorithmic traffic)
        return "hbm", th * esz * (2 * w.d_r + 2 * w.d_v), "GB/s"
    if name == "tc_causal_segment_memory":   # the write pass (key side)
        return "hbm", w.key_heads * esz * (w.d_r + w.d_v), "GB/s"
    if name == "tc_bidir_write":
        return "hbm", w.key_heads * esz * (w.d_r + w.d_v), "GB/s"
    if name == "tc_bidir_read":
        return "hbm", th * esz * (w.d_r + w.d_v), "GB/s"
    if name == "tc_responsibilities":
        if w.name.startswith("usage_"):   # the diagnostics pass: the rows read, one int32 assignment written
            return "hbm", usage_bytes(w), "GB/s"
        return "hbm", th * (esz * w.d_r + esz * w.K), "GB/s"
    if name == "usage_rows":
        return "hbm", th * (4 * w.K + 4), "GB/s"
    # backward (fp32 CUDA cores): flops of each kernel's arithmetic, in-segment (64-token) terms included
    dv1 = w.d_v + 1
    if name == "bwd_numden":        # num, den and dnd, then the segment partial Gamma_Q^T dnd
        return "alu", th * 2 * (2 * w.K * dv1 + (32 * w.K + 32 * dv1 if w.causal else 0)), "TFLOP/s"
    if name == "bwd_dgamma_q":
        return "alu", th * 2 * (w.K * dv1 + (32 * w.K + 32 * dv1 if w.causal else 0)), "TFLOP/s"
    if name == "bwd_dgamma_k_dv":
        return "alu", th * 2 * (w.K * w.d_v + w.K * dv1 + (64 * w.K + 32 * w.d_v + 32 * dv1 if w.causal else 0)), "TFLOP/s"
    if name == "bwd_param_partials":   # both sides' rows: x - mu, one product, two additions per term
        return "alu", 2 * th * w.K * w.d_r * 5, "TFLOP/s"
    if name == "bwd_dx":            # one launch covers both sides: two FMAs per term, and the softmax step
        return "alu", 2 * th * w.K * (4 * w.d_r + 2), "TFLOP/s"
    if name == "simt_responsibilities":      # one launch covers both sides (queries and keys)
        return "alu", (th + w.key_heads) * 2 * w.K * w.d_r * 3, "TFLOP/s"
    if name == "simt_small_one_launch":   # parameters, both sides' responsibilities, memory and read
        f = th * 2 * w.K * w.d_r * 3 + w.key_heads * (2 * w.K * w.d_r * 3 + 2 * w.K * (w.d_v + 1))
        return "alu", f + th * 2 * w.K * (w.d_v + 1), "TFLOP/s"
    if name == "simt_read":
        f = 2 * w.K * (w.d_v + 1)
        if w.causal:
            f += 2 * 64 * w.K + 64 * (w.d_v + 1)
        return "alu", th * f, "TFLOP/s"
    if name == "simt_segment_memory":
        return "alu", th * 2 * w.K * (w.d_v + 1), "TFLOP/s"
    if name == "decode_step":
        # the fp32 state is read and written once; q_x, k_x and v read, o written
        return "hbm", decode_bytes(w), "GB/s"
    return "hbm", 0, "GB/s"


def decode_bytes(w):
    """Algorithmic bytes of one decode step: every slice's K x (d_v + 1) fp32 state read and
    written once, plus this token's q_x, k_x, v and o."""
    esz = 2 if w.dtype == "bf16" else 4
    return w.B * w.H * (2 * 4 * w.K * (w.d_v + 1) + esz * (2 * w.d_r + 2 * w.d_v))


def traffic_per_launch(kernel, w, units=None):
    """DRAM bytes (read + write) of one launch of `kernel` on workload `w`, from the committed
    ncu summary profiles/dram_traffic.json (captured per token-head on a smaller case of the same
    kernel, scaled by the units one launch processes); None when no capture exists or any of the
    kernel's source files changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        src = os.path.join(ROOT, f)
        if not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    if h.hexdigest() != rec["sources_sha256"]:
        return None
    if rec.get("workload_shape") != [w.d_r, w.K, w.d_v, w.dtype, w.causal]:
        return None
    return rec["dram_bytes_per_token_head"] * (w.token_heads if units is None else units)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.target = None
        try:
            self.target = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.target = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.target:
            cmd += ["-i", self.target]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                smax.append(float(row[2]))
            except ValueError:
                continue
            for n, v in zip(names, row[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed
def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(w, budget_s, threads=0):
    """Time the fp64 oracle on the first n tokens of every head of batch row 0 (n sized to take
    about budget_s; exact work of the causal variant on those tokens).  Returns
    (tokens/s, cores used, description)."""
    import oracle
    host = W.to_numpy(W.make_inputs(W.scaled(w, B=1)))

    def run(n):
        sl = slice(0, n)
        t0 = time.perf_counter()
        if w.N_k:   # cross-attention: the first n queries against every key
            oracle.forward_cross(host["QX"][:, :, sl], host["KX"], host["V"], host["mu"], host["raw"],
                                 host["logits"], w.var_floor, w.eps)
            return time.perf_counter() - t0, 1
        _, used = oracle.forward(w.causal, host["QX"][:, :, sl], host["KX"][:, :, sl],
                                 host["V"][:, :, sl], host["mu"], host["raw"], host["logits"],
                                 w.var_floor, w.eps, nthreads=threads, return_threads=True)
        return time.perf_counter() - t0, used

    n = min(64, w.N)
    t, used = run(n)
    while t < budget_s / 8 and n < w.N:
        n = min(w.N, n * 4)
        t, used = run(n)
    if t < budget_s / 2 and n < w.N:
        n = min(w.N, max(n, int(n * budget_s / max(t, 1e-3))))
        t, used = run(n)
    if w.N_k:
        desc = (f"oracle cross-attention (fp64 C, one thread) on queries 0..{n - 1} against all "
                f"{w.N_k} keys of all {w.H} heads of one sequence of {w.name}")
    else:
        desc = (f"oracle (fp64 C, OpenMP over heads) on tokens 0..{n - 1} of all {w.H} heads of one "
                f"sequence of {w.name}; {'causal prefix: exact work for those tokens' if w.causal else 'bidirectional over the truncated sequence'}")
    return n / t, used, desc, n


# ----------------------------------------------------------------------------- our arm
def run_gma(args, ws, rank, local):
    from linear_latent_routing_gb300 import gma
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w0 = W.by_name(args.workload)
    over = {"seed": w0.seed + 1000 * rank}
    if args.heads:
        over["H"] = args.heads
    w = W.Workload(**{**w0.__dict__, **over})
    host = W.make_inputs(w)
    dev = {k: v.to(device) for k, v in host.items()}
    single, recompute = bool(args.single_pass), bool(args.recompute_keys)
    if (single or recompute) and not w.causal:
        raise SystemExit("--single-pass and --recompute-keys apply to causal workloads only")
    shape = gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v,
                           gma.GMA_BF16 if w.dtype == "bf16" else gma.GMA_F32, w.eps, w.var_floor,
                           flags=(gma.GMA_FLAG_SINGLE_PASS if single else 0)
                           | (gma.GMA_FLAG_RECOMPUTE_KEYS if recompute else 0))
    variant = gma.GMA_VARIANT_CAUSAL if w.causal else gma.GMA_VARIANT_BIDIRECTIONAL
    ws_n = (gma.gma_workspace_size_cross(shape, w.N_k) if w.N_k
            else gma.gma_workspace_size(shape, variant))
    workspace = torch.empty(ws_n, dtype=torch.uint8, device=device)
    O = torch.empty(w.B, w.H, w.N, w.d_v, dtype=dev["V"].dtype, device=device)
    stream = torch.cuda.Stream(device)
    sh = stream.cuda_stream
    if w.N_k:
        def fn(*a):
            return gma.gma_forward_cross(shape, w.N_k, *a[1:])
        fn.__name__ = "gma_forward_cross"
    else:
        fn = gma.gma_forward_causal if w.causal else gma.gma_forward_bidirectional
    ptrs = [dev[k].data_ptr() for k in ("QX", "KX", "V", "mu", "raw", "logits")]

    def step():
        r = fn(shape, *ptrs, O.data_ptr(), workspace.data_ptr(), ws_n, sh)
        if r != 0:
            raise gma.GmaError(r, fn.__name__)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    st = gma.gma_check_workspace(workspace.data_ptr(), sh)
    if st != 0:
        raise gma.GmaError(st, "warm-up")

    steps = args.steps
    if steps <= 0:   # auto: about 3 s of timed work, at least 20 steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(5):
                step()
            e1.record(stream)
        stream.synchronize()
        per = max(e0.elapsed_time(e1) / 5.0, 1e-3)
        steps = int(min(20000, max(20, 3000.0 / per)))

    # inputs that fit in L2 would stay there from step to step: such workloads write a buffer of
    # twice the L2 size before every timed step, outside that step's own event pair
    flush = path_bytes(w) <= L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device) if flush else None
    clocks = ClockSampler(device)
    torch.cuda.synchronize()
    barrier(ws)
    clocks.start()
    time.sleep(0.3)
    if flush:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(steps)]
        with torch.cuda.stream(stream):
            for i in range(steps):
                flush_buf.fill_(i & 0xFF)
                pairs[i][0].record(stream)
                step()
                pairs[i][1].record(stream)
    else:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                step()
            e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    total_ms = sum(a.elapsed_time(b) for a, b in pairs) if flush else e0.elapsed_time(e1)
    st = gma.gma_check_workspace(workspace.data_ptr(), sh)
    if st != 0:
        raise gma.GmaError(st, "timed region")
    # per-kernel durations from a separate pass: the events recorded around every launch would
    # keep each kernel from starting while the one ahead of it finishes
    n_bd = min(steps, 100)
    gma.gma_timing_enable(n_bd * 8 + 64)
    with torch.cuda.stream(stream):
        for i in range(n_bd):
            if flush:
                flush_buf.fill_(i & 0xFF)
            step()
    stream.synchronize()
    launches = gma.gma_timing_read(n_bd * 8 + 64)
    gma.gma_timing_enable(0)
    del flush_buf

    total_ms_max = max_over_ranks(total_ms, ws, device)
    tokens_all = w.tokens * ws * steps
    value = tokens_all / (total_ms_max / 1e3)

    # dominant kernel and its roofline
    per_kernel = {}
    for name, ms in launches:
        per_kernel.setdefault(name, []).append(ms)
    dom = max(per_kernel, key=lambda k: sum(per_kernel[k]))
    avg_ms = sum(per_kernel[dom]) / len(per_kernel[dom])
    bound, amount, unit = kernel_work(w, dom)
    if recompute and dom == "tc_causal_chunked":
        # (the recompute kernel is timed under the output pass's name; it also reads K_X)
        amount += w.token_heads * (2 if w.dtype == "bf16" else 4) * w.d_r
    pk = peaks()
    if bound == "hbm":
        achieved = amount / (avg_ms / 1e3) / 1e9
        peak = pk["hbm_gbs"]
        peak_src = f"hbm_gbs of {pk['source']}"
    elif bound == "tensor":
        achieved = amount / (avg_ms / 1e3) / 1e12
        peak = pk["bf16_tflops_sustained"]
        peak_src = f"bf16_tflops_sustained of {pk['source']}"
    else:
        achieved = amount / (avg_ms / 1e3) / 1e12
        peak = SMS * FP32_LANES_PER_SM * 2 * pk["sm_max_mhz"] * 1e6 / 1e12
        peak_src = "fp32 FMA: 152 SMs x 128 lanes x 2 flops x max SM clock"
    roofline = {"bound": bound, "kernel": dom, "achieved": round(achieved, 3),
                "peak": round(peak, 3), "unit": unit, "frac": round(achieved / peak, 4),
                "traffic": None, "avg_launch_us": round(avg_ms * 1e3, 3),
                "launches": len(per_kernel[dom]), "peak_source": peak_src}
    step_bytes = path_bytes(w)
    step_flops = path_flops(w)
    step_s = total_ms_max / steps / 1e3
    roof_s = max(step_bytes / (pk["hbm_gbs"] * 1e9), step_flops / (pk["bf16_tflops"] * 1e12))
    path_roofline = {"roofline_step_us": round(roof_s * 1e6, 3),
                     "measured_step_us": round(step_s * 1e6, 3),
                     "frac": round(roof_s / step_s, 4),
                     "alg_bytes": step_bytes, "alg_flops": step_flops}

    # (traffic records are keyed by kernel name, and the recompute kernel shares the output pass's)
    traffic = None if recompute else traffic_per_launch(dom, w)
    roofline["traffic"] = traffic

    # end to end through the C ABI with pinned host buffers.  Every step copies its own inputs from
    # pinned host memory, runs the call, and reads its output back.  Steps are pipelined over one
    # copy stream and the compute stream, with two device sets of inputs and outputs: step i + 1's
    # inputs cross the host link while step i computes, then step i's output comes back.  (The
    # copies themselves stay in one stream: copies in both directions at once ran slower on the
    # largest workload.)  A set is refilled only after its previous step finished with it.
    e2e_steps = max(4, min(steps, 12))
    pin = {k: host[k].pin_memory() for k in ("QX", "KX", "V", "mu", "raw", "logits")}
    O_host = [torch.empty(O.shape, dtype=O.dtype).pin_memory() for _ in range(2)]
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in pin)
    d2h = O_host[0].numel() * O_host[0].element_size()
    sets = [(dev, O), ({k: torch.empty_like(dev[k]) for k in pin}, torch.empty_like(O))]
    s_copy = torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        def copy_in(i):
            d, _ = sets[i % 2]
            with torch.cuda.stream(s_copy):   # (after step i - 2's output left: same stream)
                for k in pin:
                    d[k].copy_(pin[k], non_blocking=True)
                ev_in[i % 2].record(s_copy)

        copy_in(0)
        for i in range(n):
            b = i % 2
            d, o = sets[b]
            if i + 1 < n:
                copy_in(i + 1)
            stream.wait_event(ev_in[b])
            p = [d[k].data_ptr() for k in ("QX", "KX", "V", "mu", "raw", "logits")]
            r = fn(shape, *p, o.data_ptr(), workspace.data_ptr(), ws_n, sh)
            if r != 0:
                raise gma.GmaError(r, fn.__name__)
            ev_done[b].record(stream)
            s_copy.wait_event(ev_done[b])
            with torch.cuda.stream(s_copy):
                O_host[b].copy_(o, non_blocking=True)

    e2e = None
    if not args.no_e2e:
        e2e_run(2)
        torch.cuda.synchronize()
        barrier(ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_copy)
        stream.wait_event(a)
        e2e_run(e2e_steps)
        s_copy.wait_stream(stream)
        b.record(s_copy)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(a.elapsed_time(b), ws, device)
        e2e_ok = torch.equal(O_host[0], O_host[1])   # the same inputs every step: the same bits
        e2e = {"value": w.tokens * ws * e2e_steps / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "pipelined": "one copy stream and the compute stream: step i+1's inputs cross the "
                            "host link while step i computes, then step i's output comes back",
               "outputs_repeat": bool(e2e_ok)}

    if rank != 0:
        return None
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_sample(W.by_name(args.workload), args.cpu_budget)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    fam = gma.gma_kernel_family(shape, variant)
    launches_per_step = len(launches) / n_bd
    return {
        "metric": metric_for(w0), "value": value, "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": max(args.warmup, 3), "ms_per_step": total_ms_max / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded N(0,1) routing vectors and values)",
        "config": {"workload": w0.name,
                   "variant": "cross" if w.N_k else ("causal single-launch (GMA_FLAG_SINGLE_PASS)" if single
                                                     else "causal, keys recomputed (GMA_FLAG_RECOMPUTE_KEYS)"
                                                     if recompute else "causal" if w.causal else "bidirectional"),
                   "B": w.B, "H": w.H, "N": w.N, "N_k": w.keys, "d_r": w.d_r, "K": w.K, "d_v": w.d_v,
                   "eps": w.eps, "var_floor": w.var_floor,
                   "kernel_family": "tcgen05" if fam == 1 else "fp32 cuda-core",
                   "l2": ("inputs larger than L2 (%.0f MB > 129 MB), no flush"
                          % (path_bytes(w) / 1e6)) if not flush else
                         ("inputs smaller than L2 (%.1f MB): a %d MB buffer written before every "
                          "timed step, outside its event pair; value = steps / sum of the per-step "
                          "event times" % (path_bytes(w) / 1e6, 2 * L2_BYTES // 2 ** 20)),
                   "parallelism": f"replicas x{ws} (independent heads per rank)"},
        "roofline": roofline, "path_roofline": path_roofline,
        "kernels": {k: {"launches": len(v), "total_ms": round(sum(v), 4)}
                    for k, v in per_kernel.items()},
        "kernels_from_steps": n_bd,
        "gpu_launches": round(launches_per_step * steps), "launches_per_step": launches_per_step,
        "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
    }


# ----------------------------------------------------------------------------- decode
DECODE_METRIC = "GMA decode tokens/s (one new token per sequence per step), B=128,H=16,K=128,d_v=128"


def metric_for(w):
    """The headline metric for the benchmark workload; a descriptive one for the others."""
    if w.name == DEFAULT_WORKLOAD:
        return METRIC
    variant = "cross" if w.N_k else ("causal" if w.causal else "bidirectional")
    return f"GMA {variant} fwd tokens/s, {w.name} on 1 GB300"


def is_decode(w):
    return w.name.startswith("decode_")


def oracle_decode_sample(w, budget_s):
    """Time the fp64 oracle's decode step on all slices of the batch, repeated for about
    budget_s.  Returns (tokens/s, cores, description, steps)."""
    import oracle
    a = W.to_numpy(W.make_inputs(w))
    S = W.make_decode_state(w).double().numpy()
    n, t0 = 0, time.perf_counter()
    while True:
        t = n % w.N
        _, S = oracle.decode_step(a["QX"][:, :, t], a["KX"][:, :, t], a["V"][:, :, t], a["mu"],
                                  a["raw"], a["logits"], w.var_floor, w.eps, S)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    desc = (f"oracle decode step (fp64 C, one thread) over all {w.B}x{w.H} slices of {w.name}, "
            f"{n} steps")
    return w.B * n / dt, 1, desc, n


def run_decode(args, ws, rank, local):
    """One timed step = one gma_decode_step over the whole batch: every sequence takes one token.
    The state (135 MB fp32) stays on the device between steps, as a serving cache does; it is
    larger than L2, so nothing is flushed."""
    from linear_latent_routing_gb300 import gma
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w0 = W.by_name(args.workload)
    w = W.Workload(**{**w0.__dict__, "seed": w0.seed + 1000 * rank})
    host = W.make_inputs(w)
    rows = {k: [host[k][:, :, t].contiguous() for t in range(w.N)] for k in ("QX", "KX", "V")}
    drows = {k: [r.to(device) for r in rows[k]] for k in rows}
    par = {k: host[k].to(device) for k in ("mu", "raw", "logits")}
    state = W.make_decode_state(w).to(device)
    dt = gma.GMA_BF16 if w.dtype == "bf16" else gma.GMA_F32
    shape = gma.make_shape(w.B, w.H, 1, w.d_r, w.K, w.d_v, dt, w.eps, w.var_floor)
    ws_n = gma.gma_workspace_size(shape, gma.GMA_VARIANT_DECODE)
    workspace = torch.empty(ws_n, dtype=torch.uint8, device=device)
    o = torch.empty(w.B, w.H, w.d_v, dtype=host["V"].dtype, device=device)
    stream = torch.cuda.Stream(device)
    sh = stream.cuda_stream
    it = [0]

    def step(src=None):
        t = it[0] % w.N
        it[0] += 1
        q, k, v = (src or drows)["QX"][t], (src or drows)["KX"][t], (src or drows)["V"][t]
        r = gma.gma_decode_step(shape, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                par["mu"].data_ptr(), par["raw"].data_ptr(),
                                par["logits"].data_ptr(), state.data_ptr(), o.data_ptr(),
                                workspace.data_ptr(), ws_n, sh)
        if r != 0:
            raise gma.GmaError(r, "gma_decode_step")

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    steps = args.steps if args.steps > 0 else 2000
    clocks = ClockSampler(device)
    torch.cuda.synchronize()
    barrier(ws)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    st = gma.gma_check_workspace(workspace.data_ptr(), sh)
    if st != 0:
        raise gma.GmaError(st, "timed region")
    total_ms = max_over_ranks(e0.elapsed_time(e1), ws, device)
    # per-kernel durations from a separate pass: the events around each launch would keep the
    # decode kernel from starting while the parameter kernel ahead of it runs
    n_bd = min(steps, 200)
    gma.gma_timing_enable(n_bd * 4 + 64)
    with torch.cuda.stream(stream):
        for _ in range(n_bd):
            step()
    stream.synchronize()
    launches = gma.gma_timing_read(n_bd * 4 + 64)
    gma.gma_timing_enable(0)
    value = w.B * ws * steps / (total_ms / 1e3)
    per_kernel = {}
    for name, ms in launches:
        per_kernel.setdefault(name, []).append(ms)
    avg_ms = sum(per_kernel["decode_step"]) / len(per_kernel["decode_step"])
    pk = peaks()
    achieved = decode_bytes(w) / (avg_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "decode_step", "achieved": round(achieved, 3),
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": traffic_per_launch("decode_step", w, units=w.B * w.H),
                "avg_launch_us": round(avg_ms * 1e3, 3),
                "launches": len(per_kernel["decode_step"]),
                "peak_source": f"hbm_gbs of {pk['source']}"}
    step_s = total_ms / steps / 1e3
    path_roofline = {"roofline_step_us": round(decode_bytes(w) / (pk["hbm_gbs"] * 1e9) * 1e6, 3),
                     "measured_step_us": round(step_s * 1e6, 3),
                     "frac": round(decode_bytes(w) / (pk["hbm_gbs"] * 1e9) / step_s, 4),
                     "alg_bytes": decode_bytes(w)}

    # end to end: each step's q_x, k_x, v rows come from pinned host memory and o goes back
    pin = {k: [r.pin_memory() for r in rows[k]] for k in rows}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(pin[k][0].numel() * pin[k][0].element_size() for k in pin)
    d2h = o_host.numel() * o_host.element_size()
    stage = {k: [torch.empty_like(drows[k][0])] * w.N for k in drows}

    def e2e_step():
        t = it[0] % w.N
        for k in pin:
            stage[k][t].copy_(pin[k][t], non_blocking=True)
        step(stage)
        o_host.copy_(o, non_blocking=True)

    e2e = None
    if not args.no_e2e:
        e2e_steps = min(steps, 500)
        with torch.cuda.stream(stream):
            e2e_step()
        stream.synchronize()
        barrier(ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(e2e_steps):
                e2e_step()
            b.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(a.elapsed_time(b), ws, device)
        e2e = {"value": w.B * ws * e2e_steps / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}
    if rank != 0:
        return None
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_decode_sample(w0, args.cpu_budget)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    return {
        "metric": DECODE_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": max(args.warmup, 3), "ms_per_step": total_ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) rows and a seeded non-zero starting state)",
        "config": {"workload": w0.name, "variant": "decode", "B": w.B, "H": w.H, "d_r": w.d_r,
                   "K": w.K, "d_v": w.d_v, "state_bytes": 4 * w.B * w.H * w.K * (w.d_v + 1),
                   "l2": "state larger than L2 (%.0f MB > 129 MB), no flush"
                         % (4 * w.B * w.H * w.K * (w.d_v + 1) / 1e6),
                   "kernel_family": "fp32 cuda-core",
                   "parallelism": f"replicas x{ws} (independent sequences per rank)"},
        "roofline": roofline, "path_roofline": path_roofline,
        "kernels": {k: {"launches": len(v), "total_ms": round(sum(v), 4)}
                    for k, v in per_kernel.items()},
        "kernels_from_steps": n_bd,
        "gpu_launches": steps * len(launches) // n_bd, "launches_per_step": len(launches) / n_bd,
        "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
    }


# ----------------------------------------------------------------------------- usage diagnostics
def usage_bytes(w):
    """Algorithmic bytes of one diagnostics call: the routing rows read, one int32 assignment per
    token written (the per-head counts, masses and statistics are negligible)."""
    esz = 2 if w.dtype == "bf16" else 4
    return w.token_heads * (esz * w.d_r + 4)


def oracle_usage_sample(w, budget_s):
    import oracle
    a = W.to_numpy(W.make_inputs(W.scaled(w, B=1, H=1)))
    n = min(256, w.N)
    while True:
        t0 = time.perf_counter()
        oracle.usage(a["QX"][:, :, :n], a["mu"], a["raw"], a["logits"], w.var_floor)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or n >= w.N:
            break
        n = min(w.N, n * 4)
    desc = f"oracle usage diagnostics (fp64 C posterior + numpy) on tokens 0..{n - 1} of head 0 of {w.name}"
    return n / dt, 1, desc, n


def run_usage(args, ws, rank, local):
    """One step = one gma_usage call over the workload's Q_X rows (all heads)."""
    from linear_latent_routing_gb300 import gma
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w0 = W.by_name(args.workload)
    w = W.Workload(**{**w0.__dict__, "seed": w0.seed + 1000 * rank})
    host = W.make_inputs(w)
    X = host["QX"].to(device)
    par = {k: host[k].to(device) for k in ("mu", "raw", "logits")}
    shape = gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, 16, gma.GMA_BF16 if w.dtype == "bf16" else gma.GMA_F32,
                           w.eps, w.var_floor)
    ws_n = gma.gma_workspace_size(shape, gma.GMA_VARIANT_USAGE)
    workspace = torch.empty(ws_n, dtype=torch.uint8, device=device)
    out = {"assign": torch.empty(w.B, w.H, w.N, dtype=torch.int32, device=device),
           "counts": torch.empty(w.H, w.K, dtype=torch.int32, device=device),
           "mass": torch.empty(w.H, w.K, dtype=torch.float32, device=device),
           "used": torch.empty(w.H, dtype=torch.int32, device=device),
           "entropy": torch.empty(w.H, dtype=torch.float32, device=device)}
    stream = torch.cuda.Stream(device)
    sh = stream.cuda_stream

    def step(xp=None):
        r = gma.gma_usage(shape, (X if xp is None else xp).data_ptr(), par["mu"].data_ptr(), par["raw"].data_ptr(),
                          par["logits"].data_ptr(), out["assign"].data_ptr(), out["counts"].data_ptr(),
                          out["mass"].data_ptr(), out["used"].data_ptr(), out["entropy"].data_ptr(),
                          workspace.data_ptr(), ws_n, sh)
        if r != 0:
            raise gma.GmaError(r, "gma_usage")

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    steps = args.steps if args.steps > 0 else 200
    gma.gma_timing_enable(steps * 8 + 64)
    clocks = ClockSampler(device)
    torch.cuda.synchronize()
    barrier(ws)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    launches = gma.gma_timing_read(steps * 8 + 64)
    gma.gma_timing_enable(0)
    st = gma.gma_check_workspace(workspace.data_ptr(), sh)
    if st != 0:
        raise gma.GmaError(st, "timed region")
    total_ms = max_over_ranks(e0.elapsed_time(e1), ws, device)
    value = w.tokens * ws * steps / (total_ms / 1e3)
    per_kernel = {}
    for name, ms in launches:
        per_kernel.setdefault(name, []).append(ms)
    dom = max(per_kernel, key=lambda k: sum(per_kernel[k]))
    avg_ms = sum(per_kernel[dom]) / len(per_kernel[dom])
    bound, amount, unit = kernel_work(w, dom)
    pk = peaks()
    achieved = amount / (avg_ms / 1e3) / 1e9
    roofline = {"bound": bound, "kernel": dom, "achieved": round(achieved, 3), "peak": pk["hbm_gbs"],
                "unit": unit, "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
                "avg_launch_us": round(avg_ms * 1e3, 3), "launches": len(per_kernel[dom]),
                "peak_source": f"hbm_gbs of {pk['source']}"}
    step_s = total_ms / steps / 1e3
    ub = usage_bytes(w)
    path_roofline = {"roofline_step_us": round(ub / (pk["hbm_gbs"] * 1e9) * 1e6, 3),
                     "measured_step_us": round(step_s * 1e6, 3),
                     "frac": round(ub / (pk["hbm_gbs"] * 1e9) / step_s, 4), "alg_bytes": ub}
    # end to end: the rows from pinned host memory, the per-head statistics back
    pin = host["QX"].pin_memory()
    stage = torch.empty_like(X)
    res = {k: torch.empty(out[k].shape, dtype=out[k].dtype).pin_memory() for k in ("counts", "used", "entropy")}
    h2d = pin.numel() * pin.element_size()
    d2h = sum(res[k].numel() * res[k].element_size() for k in res)

    def e2e_step():
        stage.copy_(pin, non_blocking=True)
        step(stage)
        for k in res:
            res[k].copy_(out[k], non_blocking=True)

    e2e = None
    if not args.no_e2e:
        n_e = min(steps, 20)
        with torch.cuda.stream(stream):
            e2e_step()
        stream.synchronize()
        barrier(ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(n_e):
                e2e_step()
            b.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(a.elapsed_time(b), ws, device)
        e2e = {"value": w.tokens * ws * n_e / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e}
    if rank != 0:
        return None
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_usage_sample(w0, args.cpu_budget)
        cpu = {"value": v / w.H, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": desc + f"; divided by the {w.H} heads a token carries"}
    return {
        "metric": f"GMA usage diagnostics tokens/s, {w0.name} on 1 GB300", "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": total_ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) routing rows)",
        "config": {"workload": w0.name, "variant": "usage", "B": w.B, "H": w.H, "N": w.N, "d_r": w.d_r,
                   "K": w.K, "kernel_family": "tcgen05" if gma.gma_kernel_family(shape, gma.GMA_VARIANT_USAGE) == 1
                   else "fp32 cuda-core",
                   "l2": "fp32 responsibilities (537 MB) larger than L2, no flush",
                   "parallelism": f"replicas x{ws}"},
        "roofline": roofline, "path_roofline": path_roofline,
        "kernels": {k: {"launches": len(v), "total_ms": round(sum(v), 4)} for k, v in per_kernel.items()},
        "gpu_launches": len(launches), "launches_per_step": len(launches) / steps,
        "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
    }


# ----------------------------------------------------------------------------- backward pass
def backward_bytes(w):
    """Algorithmic bytes of one backward call: Q_X, K_X, V and dO read, dQ_X, dK_X, dV written."""
    esz = 2 if w.dtype == "bf16" else 4
    return w.token_heads * esz * (4 * w.d_r + 3 * w.d_v)


def _bwd_dO(w):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed) + 2024)
    d = torch.randn(w.B, w.H, w.N, w.d_v, generator=g, dtype=torch.float32)
    return d.to(torch.bfloat16) if w.dtype == "bf16" else d


def oracle_backward_sample(w, budget_s):
    import oracle
    ws_ = W.scaled(w, B=1, H=1)
    a = W.to_numpy(W.make_inputs(ws_))
    dO = _bwd_dO(w)[:1, :1].float().numpy()
    n = 64
    while True:
        t0 = time.perf_counter()
        oracle.backward(w.causal, a["QX"][:, :, :n], a["KX"][:, :, :n], a["V"][:, :, :n], a["mu"], a["raw"],
                        a["logits"], w.var_floor, w.eps, dO[:, :, :n])
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or n >= w.N:
            break
        n = min(w.N, n * 2)
    desc = (f"oracle backward (fp64, explicit affinity form) on tokens 0..{n - 1} of one head of {w.name}; "
            f"its work grows as N^2, so longer prefixes would be slower per token")
    return n / dt, 1, desc, n


def run_backward(args, ws, rank, local):
    """One step = one gma_backward call (the whole layer's gradients) on the workload."""
    from linear_latent_routing_gb300 import gma
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w0 = W.by_name(args.workload)
    w = W.Workload(**{**w0.__dict__, "seed": w0.seed + 1000 * rank})
    host = W.make_inputs(w)
    host["dO"] = _bwd_dO(w)
    dev = {k: v.to(device) for k, v in host.items()}
    shape = gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v, gma.GMA_BF16 if w.dtype == "bf16" else gma.GMA_F32,
                           w.eps, w.var_floor)
    ws_n = gma.gma_workspace_size(shape, gma.GMA_VARIANT_BACKWARD)
    workspace = torch.empty(ws_n, dtype=torch.uint8, device=device)
    outs = [torch.empty_like(dev["QX"]), torch.empty_like(dev["KX"]), torch.empty_like(dev["V"]),
            torch.empty_like(dev["mu"]), torch.empty_like(dev["raw"]), torch.empty_like(dev["logits"])]
    stream = torch.cuda.Stream(device)
    sh = stream.cuda_stream

    def step(src=None):
        d = src or dev
        r = gma.gma_backward(shape, 1 if w.causal else 0, *[d[k].data_ptr() for k in ("QX", "KX", "V")],
                             *[dev[k].data_ptr() for k in ("mu", "raw", "logits")], d["dO"].data_ptr(),
                             *[t.data_ptr() for t in outs], workspace.data_ptr(), ws_n, sh)
        if r != 0:
            raise gma.GmaError(r, "gma_backward")

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    steps = args.steps if args.steps > 0 else 50
    gma.gma_timing_enable(steps * 16 + 64)
    clocks = ClockSampler(device)
    torch.cuda.synchronize()
    barrier(ws)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    launches = gma.gma_timing_read(steps * 16 + 64)
    gma.gma_timing_enable(0)
    st = gma.gma_check_workspace(workspace.data_ptr(), sh)
    if st != 0:
        raise gma.GmaError(st, "timed region")
    total_ms = max_over_ranks(e0.elapsed_time(e1), ws, device)
    value = w.tokens * ws * steps / (total_ms / 1e3)
    per_kernel = {}
    for name, ms in launches:
        per_kernel.setdefault(name, []).append(ms)
    dom = max(per_kernel, key=lambda k: sum(per_kernel[k]))
    avg_ms = sum(per_kernel[dom]) / len(per_kernel[dom])
    bound, amount, unit = kernel_work(w, dom)
    pk = peaks()
    if bound == "alu":
        achieved = amount / (avg_ms / 1e3) / 1e12
        peak = SMS * FP32_LANES_PER_SM * 2 * pk["sm_max_mhz"] * 1e6 / 1e12
        src = "fp32 FMA: 152 SMs x 128 lanes x 2 flops x max SM clock"
    else:
        achieved = amount / (avg_ms / 1e3) / 1e9
        peak = pk["hbm_gbs"]
        src = f"hbm_gbs of {pk['source']}"
    roofline = {"bound": bound, "kernel": dom, "achieved": round(achieved, 3), "peak": round(peak, 3),
                "unit": unit, "frac": round(achieved / peak, 4), "traffic": None,
                "avg_launch_us": round(avg_ms * 1e3, 3), "launches": len(per_kernel[dom]), "peak_source": src}
    bb = backward_bytes(w)
    step_s = total_ms / steps / 1e3
    path_roofline = {"roofline_step_us": round(bb / (pk["hbm_gbs"] * 1e9) * 1e6, 3),
                     "measured_step_us": round(step_s * 1e6, 3),
                     "frac": round(bb / (pk["hbm_gbs"] * 1e9) / step_s, 4), "alg_bytes": bb}
    pin = {k: host[k].pin_memory() for k in ("QX", "KX", "V", "dO")}
    stage = {k: torch.empty_like(dev[k]) for k in pin}
    res = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in res)

    def e2e_step():
        for k in pin:
            stage[k].copy_(pin[k], non_blocking=True)
        step(stage)
        for a, b in zip(res, outs):
            a.copy_(b, non_blocking=True)

    e2e = None
    if not args.no_e2e:
        n_e = min(steps, 10)
        with torch.cuda.stream(stream):
            e2e_step()
        stream.synchronize()
        barrier(ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(n_e):
                e2e_step()
            b.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(a.elapsed_time(b), ws, device)
        e2e = {"value": w.tokens * ws * n_e / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e}
    if rank != 0:
        return None
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_backward_sample(w0, args.cpu_budget)
        cpu = {"value": v / w.H, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": desc + f"; divided by the {w.H} heads a token carries"}
    return {
        "metric": f"GMA backward tokens/s, {w0.name} on 1 GB300", "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": total_ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 (bf16 in/out)",
        "data": "synthetic (seeded N(0,1) rows, values and output gradients)",
        "config": {"workload": w0.name, "variant": "backward, causal" if w.causal else "backward, bidirectional",
                   "B": w.B, "H": w.H, "N": w.N, "d_r": w.d_r, "K": w.K, "d_v": w.d_v,
                   "kernel_family": "fp32 cuda-core", "l2": "not flushed (workspace > L2)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": roofline, "path_roofline": path_roofline,
        "kernels": {k: {"launches": len(v), "total_ms": round(sum(v), 4)} for k, v in per_kernel.items()},
        "gpu_launches": len(launches), "launches_per_step": len(launches) / steps,
        "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
    }


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, ws, rank):
    if rank != 0:
        return None
    w = W.by_name(args.workload)
    steps = args.steps if args.steps > 0 else 5
    warm = max(args.warmup, 3)
    per_step_budget = min(5.0, 150.0 / (steps + warm))
    if is_decode(w):
        return run_reference_decode(args, w, ws, steps, warm, per_step_budget)
    if w.name.startswith("usage_"):
        return run_reference_usage(args, w, ws, steps, warm, per_step_budget)
    if w.name.startswith("backward_"):
        return run_reference_backward(args, w, ws, steps, warm, per_step_budget)
    rate, cores, desc, n = oracle_sample(w, per_step_budget)
    import oracle
    host = W.to_numpy(W.make_inputs(W.scaled(w, B=1)))
    sl = slice(0, n)

    def one():
        if w.N_k:
            oracle.forward_cross(host["QX"][:, :, sl], host["KX"], host["V"], host["mu"], host["raw"],
                                 host["logits"], w.var_floor, w.eps)
            return
        oracle.forward(w.causal, host["QX"][:, :, sl], host["KX"][:, :, sl], host["V"][:, :, sl],
                       host["mu"], host["raw"], host["logits"], w.var_floor, w.eps)

    for _ in range(warm):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    dt = time.perf_counter() - t0
    value = n * steps / dt
    return {
        "impl": "reference", "metric": metric_for(w), "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": steps, "warmup": warm, "ms_per_step": dt / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded), truncated sample",
        "config": {"workload": w.name,
                   "variant": "cross" if w.N_k else ("causal" if w.causal else "bidirectional"),
                   "B": w.B, "H": w.H, "N": w.N, "N_k": w.keys, "d_r": w.d_r, "K": w.K, "d_v": w.d_v},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_backward(args, w, ws, steps, warm, per_step_budget):
    rates = []
    for i in range(warm + steps):
        rate, cores, desc, n = oracle_backward_sample(w, per_step_budget)
        if i >= warm:
            rates.append(rate)
    value = sum(rates) / len(rates) / w.H
    return {
        "impl": "reference", "metric": f"GMA backward tokens/s, {w.name} on 1 GB300",
        "value": value, "unit": UNIT, "n_gpus": ws, "steps": steps, "warmup": warm,
        "ms_per_step": w.tokens / value * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded), truncated sample",
        "config": {"workload": w.name, "variant": "backward", "B": w.B, "H": w.H, "N": w.N, "d_r": w.d_r,
                   "K": w.K, "d_v": w.d_v},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc + f"; divided by the {w.H} heads a token carries"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_usage(args, w, ws, steps, warm, per_step_budget):
    rates = []
    for i in range(warm + steps):
        rate, cores, desc, n = oracle_usage_sample(w, per_step_budget)
        if i >= warm:
            rates.append(rate)
    value = sum(rates) / len(rates) / w.H   # a token carries H heads
    return {
        "impl": "reference", "metric": f"GMA usage diagnostics tokens/s, {w.name} on 1 GB300",
        "value": value, "unit": UNIT, "n_gpus": ws, "steps": steps, "warmup": warm,
        "ms_per_step": w.tokens / value * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded), truncated sample",
        "config": {"workload": w.name, "variant": "usage", "B": w.B, "H": w.H, "N": w.N, "d_r": w.d_r,
                   "K": w.K},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc + f"; divided by the {w.H} heads a token carries"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_decode(args, w, ws, steps, warm, per_step_budget):
    for _ in range(warm):
        oracle_decode_sample(w, per_step_budget / 4)
    t0 = time.perf_counter()
    n_all = 0
    for _ in range(steps):
        _, cores, desc, n = oracle_decode_sample(w, per_step_budget)
        n_all += n
    dt = time.perf_counter() - t0
    value = w.B * n_all / dt
    return {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": steps, "warmup": warm, "ms_per_step": dt / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": w.name, "variant": "decode", "B": w.B, "H": w.H, "d_r": w.d_r,
                   "K": w.K, "d_v": w.d_v},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: about 3 s of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[x.name for x in W.ALL_WORKLOADS + (W.DECODE,)])
    ap.add_argument("--impl", default="gma", choices=["gma", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU work for the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) leg")
    ap.add_argument("--heads", type=int, default=0,
                    help="profiling only: run the workload with this many heads instead")
    ap.add_argument("--single-pass", action="store_true",
                    help="causal workloads: time the single-launch variant (GMA_FLAG_SINGLE_PASS)")
    ap.add_argument("--recompute-keys", action="store_true",
                    help="causal workloads: time the variant that recomputes Gamma_K (GMA_FLAG_RECOMPUTE_KEYS)")
    args = ap.parse_args()

    if args.impl == "reference":
        ws, rank, _ = dist_setup("gloo") if int(os.environ.get("WORLD_SIZE", "1")) > 1 else (1, 0, 0)
        out = run_reference(args, ws, rank)
    else:
        from linear_latent_routing_gb300 import build
        build.build()
        ws, rank, local = dist_setup("nccl")
        w = W.by_name(args.workload)
        runner = (run_decode if is_decode(w) else run_usage if w.name.startswith("usage_")
                  else run_backward if w.name.startswith("backward_") else run_gma)
        out = runner(args, ws, rank, local)
    if out is not None:
        print(json.dumps(out), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
