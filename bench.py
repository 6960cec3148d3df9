"""Benchmark: RMSNorm backward on GB300, one JSON line on stdout (rank 0).

Default workload: plain RMSNorm backward, bf16, M=4096, N=4096, eps=1e-6,
rstd from this library's forward; a step is one public backward call
(row pass + cross-row weight-gradient reduction + fp32->bf16 cast), timed
with CUDA events on the launching stream after the L2 has been flushed
(outside the event pair) by writing a buffer twice the L2 size and then
reading another one of that size: L2 then holds none of the step's data and
no dirty lines whose write-back would land inside the timed call.

  value      algorithmic bytes / time, GB/s (whole job: summed over ranks,
             divided by the slowest rank's time)
  roofline   the row-pass kernel alone (events the library records around
             it), against the measured HBM copy bandwidth
  e2e        the same metric with host (pinned) inputs copied in and dx,
             dweight copied out inside every timed step
  cpu_baseline  the fp64 CPU oracle on the host cores, same workload
  steady     context only: back-to-back calls in a CUDA graph over problem
             sets whose dx buffers alone exceed twice the L2, one event pair
             around all of them (what a loop of backward calls sustains)

`--impl reference` times the CPU oracle as the reference arm.
Multi-GPU (torchrun): every rank runs an independent replica (the rows of
this workload shard with no exchange but the weight-gradient sum, which a
training framework's gradient all-reduce already performs).
"""
import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s (% of peak), RMSNorm & fused-add bwd, 1 GB300"
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "bwd_row_kernel_bf16_4096x4096.md")
KERNEL_SOURCES = [os.path.join(ROOT, "rmsnorm_backward_bwd_gb300", "csrc", f)
                  for f in ("bwd_row.cu", "row_math.cuh", "common.cuh")]


def kernel_source_hash():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The row-pass kernel each engine launches (from the plan string).
ENGINE_KERNELS = {"row": "bwd_row_kernel", "cluster": "bwd_cluster_kernel",
                  "generic staged": "bwd_stage_kernel",
                  "generic phase": "bwd_phase_kernel", "generic realign": "bwd_realign_kernel",
                  "generic vec": "bwd_generic_vec_kernel", "generic": "bwd_generic_kernel"}


def row_pass_kernel(plan):
    engine = plan.split("engine=", 1)[1].split(" threads=")[0].split(" rows=")[0] if plan else ""
    engine = engine.split(" cpt=")[0].split(" csize=")[0].split(" cpb=")[0]
    return ENGINE_KERNELS.get(engine, engine)


def ncu_traffic(workload):
    """DRAM bytes per launch of the row-pass kernel from the committed ncu
    summary, if that summary covers this workload and was taken on the
    current kernel source."""
    if workload != "plain_4096":
        return None
    try:
        with open(PROFILE_SUMMARY) as f:
            text = f.read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9,]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_tr.group(1).replace(",", ""))


class L2Flush:
    """Write a 2x-L2 buffer, then read another 2x-L2 buffer."""

    def __init__(self, l2_bytes, dev):
        import torch
        self.wbuf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        self.rbuf = torch.ones(2 * l2_bytes // 4, dtype=torch.float32, device=dev)
        self.mib = (2 * l2_bytes) >> 20

    def __call__(self):
        self.wbuf.zero_()
        self.rbuf.sum()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a window."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        inwin = [p for ts, p in rows if any(a - 0.15 <= ts <= b + 0.15 for a, b in self.windows)]
        use = inwin if inwin else rows
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = sorted(x for x in (num(p[2]) for p in use) if x is not None)
        mx = [x for x in (num(p[3]) for p in use) if x is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if p[6 + i] == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use), "samples_in_window": len(inwin)}


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, ws):
    """The largest value over all ranks (every rank gets it)."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank, ws, slowest_ms):
    """Replicas: every rank moves bytes_per_rank; the job takes as long as
    its slowest rank."""
    return bytes_per_rank * ws / (slowest_ms * 1e-3) / 1e9


def synth_bytes(case):
    from rmsnorm_backward_bwd_gb300 import synth
    if case.name.startswith("layernorm"):
        return synth.ln_algorithmic_bytes(case.M, case.N, case.dtype, True, True)
    return synth.algorithmic_bytes(case.M, case.N, case.dtype, case.with_dres, True)


def workload_case(name):
    from rmsnorm_backward_bwd_gb300 import synth
    table = {"plain_4096": synth.PLAIN_4096, "fused_4096": synth.FUSED_4096,
             "fused_4096_nodres": synth.FUSED_4096_NODRES, "plain_16384x8192": synth.LARGE_PLAIN,
             "fused_16384x8192": synth.LARGE_FUSED, "layernorm_4096": synth.LN_4096,
             "layernorm_16384x8192": synth.LN_LARGE,
             "plain_4096x32768": synth.LONG_ROWS, "plain_4096x4095": synth.UNALIGNED_ROWS,
             "plain_4096x12290": synth.UNALIGNED_WIDE_ROWS}
    return table[name]


class Problem:
    """Device-resident inputs/outputs of one backward case, plus the call."""

    def __init__(self, case, dev):
        import torch
        import rmsnorm_backward_bwd_gb300 as rn
        from rmsnorm_backward_bwd_gb300 import synth
        self.case = case
        inp = synth.make_inputs(case, device=str(dev))
        g = inp["gamma"]
        if case.fused:
            # the saved `added` and its rstd come from the fused forward
            _, self.x, self.rstd = rn.fused_add_rmsnorm_fwd(inp["x"], inp["residual"], g, case.eps)
            del inp["residual"]
        else:
            self.x = inp["x"]
            _, self.rstd = rn.rmsnorm_fwd(self.x, g, case.eps)
        self.g, self.dy, self.dres = g, inp["dy"], inp.get("dres")
        self.dx = torch.empty_like(self.x)
        self.dw32 = torch.empty(case.N, dtype=torch.float32, device=dev)
        self.dw = torch.empty(case.N, dtype=self.x.dtype, device=dev)
        self.ws = rn.bwd_workspace(case.M, case.N, self.x.dtype, dev)
        self.bytes = synth.algorithmic_bytes(case.M, case.N, case.dtype, case.with_dres, True)
        s = synth.ELEM_BYTES[case.dtype]
        # the row pass alone: read x|added, dy, [dres], gamma, rstd; write dx
        self.row_pass_bytes = (case.M * case.N * s * (4 if case.with_dres else 3)
                               + case.N * s + 4 * case.M)
        torch.cuda.synchronize()

    def call(self):
        import rmsnorm_backward_bwd_gb300 as rn
        if self.case.fused:
            rn.fused_add_rmsnorm_bwd(self.x, self.g, self.dy, self.rstd, self.dres, dx=self.dx,
                                     dweight_f32=self.dw32, dweight=self.dw, workspace=self.ws)
        else:
            rn.rmsnorm_bwd(self.x, self.g, self.dy, self.rstd, dx=self.dx, dweight_f32=self.dw32,
                           dweight=self.dw, workspace=self.ws)


class LnProblem:
    """Device-resident inputs/outputs of one LayerNorm backward, plus the call
    (mean and rstd from the GPU LayerNorm forward)."""

    def __init__(self, case, dev):
        import torch
        import rmsnorm_backward_bwd_gb300 as rn
        from rmsnorm_backward_bwd_gb300 import synth
        self.case = case
        inp = synth.make_ln_inputs(case, device=str(dev))
        self.x, self.g, self.dy = inp["x"], inp["gamma"], inp["dy"]
        _, self.mean, self.rstd = rn.layernorm_fwd(self.x, self.g, inp["beta"], case.eps)
        N = case.N
        self.dx = torch.empty_like(self.x)
        self.dg32 = torch.empty(N, dtype=torch.float32, device=dev)
        self.db32 = torch.empty(N, dtype=torch.float32, device=dev)
        self.dg = torch.empty(N, dtype=self.x.dtype, device=dev)
        self.db = torch.empty(N, dtype=self.x.dtype, device=dev)
        self.ws = rn.layernorm_bwd_workspace(case.M, N, self.x.dtype, dev)
        self.bytes = synth.ln_algorithmic_bytes(case.M, N, case.dtype, True, True)
        s = synth.ELEM_BYTES[case.dtype]
        self.row_pass_bytes = case.M * N * s * 3 + N * s + 8 * case.M
        torch.cuda.synchronize()

    def call(self):
        import rmsnorm_backward_bwd_gb300 as rn
        rn.layernorm_bwd(self.x, self.g, self.dy, self.mean, self.rstd, dx=self.dx,
                         dgamma_f32=self.dg32, dbeta_f32=self.db32, dgamma=self.dg,
                         dbeta=self.db, workspace=self.ws)


def launches_per_call(plan):
    if "dw=atomic" in plan:
        return 3  # zero, row pass, cast
    return 2      # row pass, finalize (+cast)


def time_calls(prob, steps, warmup, flush, ws, sampler=None, kernel_events=False):
    """Per-call device time (ms) with an L2 flush before each call."""
    import torch
    from rmsnorm_backward_bwd_gb300 import native
    for _ in range(warmup):
        flush()
        prob.call()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)] if kernel_events else None
    if kev:
        # torch creates the CUDA event on its first record: do that here, so
        # that the handles passed to the library are real events
        for a, b in kev:
            a.record(st)
            b.record(st)
        torch.cuda.synchronize()
    t0 = time.time()
    for i in range(steps):
        flush()
        if kev:
            native.lib().rn_set_profile_events(kev[i][0].cuda_event, kev[i][1].cuda_event)
        ev[i][0].record(st)
        prob.call()
        ev[i][1].record(st)
    if kev:
        native.lib().rn_set_profile_events(None, None)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(ws)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(t0, t1)
    call_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in kev] if kev else None
    return call_ms, kern_ms, t1 - t0


def time_steady(case, dev, steps, ws, l2_bytes):
    """Device time per call of back-to-back calls, as a loop of backward calls
    runs them: one CUDA graph holds 8 rounds of calls over R problem sets, and
    one event pair brackets all replays. R is the smallest count whose dx
    buffers alone exceed twice the L2: the inputs are streamed with an
    evict-first policy, so the outputs are what stays in L2 longest, and a
    call must find neither its inputs nor its last dx there. Unlike the
    flushed per-call timing, the write-back of earlier calls' dx falls inside
    the timed region, and no event sits between calls.
    Returns (ms per call, R, calls timed, plan)."""
    import torch
    from rmsnorm_backward_bwd_gb300 import native
    probs = [Problem(case, dev)]
    dx_bytes = probs[0].dx.numel() * probs[0].dx.element_size()
    while len(probs) * dx_bytes <= 2 * l2_bytes:
        probs.append(Problem(case, dev))
    R = len(probs)
    for p in probs:   # plan and workspace set up outside the capture
        p.call()
    torch.cuda.synchronize()
    per_graph = 8 * R
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(per_graph):
            probs[i % R].call()
    plan = native.last_plan()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    reps = max(3, steps // per_graph)
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * per_graph)
    del graph, probs
    torch.cuda.empty_cache()
    return ms, R, reps * per_graph, plan


def time_e2e(prob, steps, warmup, ws):
    """The same public call with its inputs in pinned host memory: every step
    copies that step's inputs (x|added, gamma, dy, rstd, [dres]) host->device,
    runs the backward and copies dx + dweight device->host, all inside the
    timed region. Steps are pipelined the way an input stream would be: two
    device buffer sets and three streams (copy in, compute, copy out), so the
    copy-in of step i+1 and the copy-out of step i-1 overlap the backward of
    step i. Returns (ms per step, host->device bytes, device->host bytes)."""
    import torch
    import rmsnorm_backward_bwd_gb300 as rn
    c = prob.case
    names = ["x", "g", "dy", "rstd"] + (["dres"] if prob.dres is not None else [])
    host = {k: getattr(prob, k).cpu().pin_memory() for k in names}
    out_dx = torch.empty(prob.dx.shape, dtype=prob.dx.dtype).pin_memory()
    out_dw = torch.empty(prob.dw.shape, dtype=prob.dw.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_dx.numel() * out_dx.element_size() + out_dw.numel() * out_dw.element_size()

    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(comp):
        ws_comp = rn.bwd_workspace(c.M, c.N, prob.x.dtype, prob.x.device)
    sets = []
    for _ in range(2):
        d = {k: torch.empty_like(getattr(prob, k)) for k in names}
        d["dx"] = torch.empty_like(prob.dx)
        d["dw32"] = torch.empty_like(prob.dw32)
        d["dw"] = torch.empty_like(prob.dw)
        sets.append(d)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("inp", "done", "out")}
    torch.cuda.synchronize()

    def step(i):
        b, d = i % 2, sets[i % 2]
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(ev["done"][b])   # the backward of step i-2 read these inputs
            for k in names:
                d[k].copy_(host[k], non_blocking=True)
            ev["inp"][b].record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(ev["inp"][b])
            if i >= 2:
                comp.wait_event(ev["out"][b])  # step i-2's outputs have been copied out
            if c.fused:
                rn.fused_add_rmsnorm_bwd(d["x"], d["g"], d["dy"], d["rstd"], d.get("dres"),
                                         dx=d["dx"], dweight_f32=d["dw32"], dweight=d["dw"],
                                         workspace=ws_comp)
            else:
                rn.rmsnorm_bwd(d["x"], d["g"], d["dy"], d["rstd"], dx=d["dx"],
                               dweight_f32=d["dw32"], dweight=d["dw"], workspace=ws_comp)
            ev["done"][b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev["done"][b])
            out_dx.copy_(d["dx"], non_blocking=True)
            out_dw.copy_(d["dw"], non_blocking=True)
            ev["out"][b].record(down)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(ws)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(up)
    for i in range(steps):
        step(i)
    z.record(down)
    torch.cuda.synchronize()
    barrier(ws)
    # the pipelined steps produced the same dx as the device-resident call
    if not torch.equal(out_dx, prob.dx.cpu()):
        raise RuntimeError("end-to-end steps disagree with the device-resident call")
    return a.elapsed_time(z) / steps, h2d, d2h


# The shape table of the FlyDSL PR #854 backward benchmark ("Summary" table):
# (op, M, N, dtype). The fused-add rows here pass a residual_out gradient.
PAGES_AUTOGRAD_SHAPES = [(op, M, N, dt) for (M, N, dt) in
                         ((1, 4096, "bf16"), (128, 4096, "bf16"), (4096, 4096, "bf16"),
                          (512, 2048, "bf16"), (512, 3000, "f32"), (1024, 8192, "bf16"))
                         for op in ("rmsnorm_bwd", "fused_add_bwd")]


def autograd_pages_table(dev, steps=100, warmup=10):
    """The public-autograd backward at the pages' benchmark shapes, this
    package against torch eager on the same GPU, timed the pages' way: hot
    cache, `warmup` calls, then the mean of `steps` calls between CUDA events;
    backward allocations, the dweight zero and the cast are inside. Gradients
    are compared before timing."""
    import numpy as np
    import torch
    from rmsnorm_backward_bwd_gb300.synth import Case
    rows = []
    for op, M, N, dt in PAGES_AUTOGRAD_SHAPES:
        case = Case(op, M, N, dt, fused=op == "fused_add_bwd", with_dres=op == "fused_add_bwd")
        res = {"op": op, "M": M, "N": N, "dtype": dt}
        grads = {}
        for impl in ("ours", "torch_eager"):
            outs, ins, gos = autograd_problem(case, dev, impl)
            grads[impl] = [t.float() for t in torch.autograd.grad(outs, ins, gos, retain_graph=True)]
            for _ in range(warmup):
                torch.autograd.grad(outs, ins, gos, retain_graph=True)
            torch.cuda.synchronize()
            st = torch.cuda.current_stream()
            ts = []
            for _ in range(steps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(st)
                torch.autograd.grad(outs, ins, gos, retain_graph=True)
                b.record(st)
                ts.append((a, b))
            torch.cuda.synchronize()
            res[impl + "_us"] = round(float(np.mean([a.elapsed_time(b) for a, b in ts])) * 1e3, 2)
            del outs, ins, gos
        res["max_rel_diff"] = float("%.3g" % max(
            float((u - v).abs().max() / v.abs().max().clamp_min(1e-30))
            for u, v in zip(grads["ours"], grads["torch_eager"])))
        res["torch_over_ours"] = round(res["torch_eager_us"] / res["ours_us"], 2)
        rows.append(res)
        del grads
        torch.cuda.empty_cache()
    return rows


def time_forwards(dev, flush, steps, warmup, peak):
    """The forwards (RMSNorm, fused-add, LayerNorm; bf16) at 4096x4096 and
    16384x8192, and on rows that are not 16-byte multiples at 4096x4095 and
    16384x8190: mean device time per call with an L2 flush before each, the
    algorithmic bytes (inputs read once, outputs and statistics written once)
    over that time, the plan, and torch eager on the same inputs beside them."""
    import numpy as np
    import torch
    import rmsnorm_backward_bwd_gb300 as rn
    from rmsnorm_backward_bwd_gb300 import synth
    from rmsnorm_backward_bwd_gb300.synth import Case

    def timed(fn):
        for _ in range(warmup):
            flush()
            fn()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            flush()
            a.record(st)
            fn()
            b.record(st)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3

    rows = []
    from rmsnorm_backward_bwd_gb300 import native
    for M, N in ((4096, 4096), (16384, 8192), (4096, 4095), (16384, 8190)):
        inp = synth.make_inputs(Case("forward", M, N, "bf16", fused=True), device=str(dev))
        x, r, g = inp["x"], inp["residual"], inp["gamma"]
        y, ro = torch.empty_like(x), torch.empty_like(x)
        mean = torch.empty(M, dtype=torch.float32, device=dev)
        rstd = torch.empty(M, dtype=torch.float32, device=dev)
        s = 2
        plain = M * N * s * 2 + N * s + 4 * M
        cases = [
            ("rmsnorm_fwd", plain, lambda: rn.rmsnorm_fwd(x, g, 1e-6, y=y, rstd=rstd)),
            ("fused_add_rmsnorm_fwd", M * N * s * 4 + N * s + 4 * M,
             lambda: rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6, out=y, residual_out=ro, rstd=rstd)),
            ("layernorm_fwd (bias)", plain + N * s + 4 * M,
             lambda: rn.layernorm_fwd(x, g, g, 1e-5, y=y, mean=mean, rstd=rstd)),
        ]
        for name, nbytes, fn in cases:
            us = timed(fn)
            rows.append({"workload": "%s bf16 M=%d N=%d" % (name, M, N), "us_per_call": round(us, 2),
                         "GBps": round(nbytes / us / 1e3, 1),
                         "pct_of_peak": round(100 * nbytes / us / 1e3 / peak, 1),
                         "plan": native.last_plan()})
        us = timed(lambda: torch.nn.functional.rms_norm(x, (N,), g, 1e-6))
        rows.append({"workload": "torch eager rms_norm bf16 M=%d N=%d" % (M, N),
                     "us_per_call": round(us, 2)})
        us = timed(lambda: torch.nn.functional.layer_norm(x, (N,), g, g, 1e-5))
        rows.append({"workload": "torch eager layer_norm (bias) bf16 M=%d N=%d" % (M, N),
                     "us_per_call": round(us, 2)})
        del inp, x, r, g, y, ro
        torch.cuda.empty_cache()
    return rows


def autograd_problem(case, dev, impl):
    """Forward graph of one case built once (outside timing): returns
    (outputs, inputs, grad_outputs) for torch.autograd.grad. impl "ours" uses
    this package's autograd wrappers, "torch_eager" torch's own rms_norm."""
    import torch
    import rmsnorm_backward_bwd_gb300 as rn
    from rmsnorm_backward_bwd_gb300 import synth
    if case.name.startswith("layernorm"):
        inp = synth.make_ln_inputs(case, device=str(dev))
        x, w, b = (inp[k].requires_grad_() for k in ("x", "gamma", "beta"))
        if impl == "ours":
            y = rn.layernorm(x, w, b, case.eps)
        else:
            y = torch.nn.functional.layer_norm(x, (case.N,), w, b, case.eps)
        return (y,), (x, w, b), (inp["dy"],)
    inp = synth.make_inputs(case, device=str(dev))
    x = inp["x"].requires_grad_()
    w = inp["gamma"].requires_grad_()
    if not case.fused:
        if impl == "ours":
            y = rn.rmsnorm(x, w, case.eps)
        else:
            y = torch.nn.functional.rms_norm(x, (case.N,), w, case.eps)
        return (y,), (x, w), (inp["dy"],)
    r = inp["residual"].requires_grad_()
    if impl == "ours":
        out, res_out = rn.fused_add_rmsnorm(x, r, w, case.eps)
    else:
        res_out = x + r
        out = torch.nn.functional.rms_norm(res_out, (case.N,), w, case.eps)
    return (out, res_out), (x, r, w), (inp["dy"], inp["dres"])


def time_autograd(graph, steps, warmup, flush, queued=False):
    """Mean time (ms) between CUDA events around torch.autograd.grad over the
    saved graph, with an L2 flush before each call; output allocation, the
    fp32 dweight zero and the cast are inside the timed region.

    queued=False: the host issues the call right after the flush, so host-side
    time (autograd engine, Python, launches) shows wherever it exceeds the GPU
    work. queued=True: a GPU sleep of ~0.5 ms after the flush keeps the device
    busy while the host issues the whole backward, so the events bracket the
    device work alone."""
    import numpy as np
    import torch
    outs, ins, gos = graph
    for _ in range(warmup):
        flush()
        torch.autograd.grad(outs, ins, gos, retain_graph=True)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()
        if queued:
            torch.cuda._sleep(1_000_000)
        a.record(st)
        torch.autograd.grad(outs, ins, gos, retain_graph=True)
        b.record(st)
        if queued:
            b.synchronize()   # keep the host from running ahead of the sleep
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in ev]))


def oracle_rate(case, seconds, nthreads=0):
    """fp64 CPU oracle on the case's full problem, repeated for ~`seconds`."""
    import numpy as np
    import torch
    import oracle
    from rmsnorm_backward_bwd_gb300 import synth
    inp = synth.make_inputs(case)
    g = inp["gamma"].to(torch.float64).numpy()
    dy = inp["dy"].to(torch.float64).numpy()
    if case.fused:
        _, x, rstd = oracle.fused_add_rmsnorm_fwd(inp["x"].to(torch.float64).numpy(),
                                                  inp["residual"].to(torch.float64).numpy(), g,
                                                  np.float32(case.eps), case.dtype, nthreads)
    else:
        x = inp["x"].to(torch.float64).numpy()
        _, rstd = oracle.rmsnorm_fwd(x, g, np.float32(case.eps), nthreads)
    rstd = oracle.round_to(rstd, "f32")
    dres = inp["dres"].to(torch.float64).numpy() if "dres" in inp else None
    cores = oracle.max_threads() if nthreads <= 0 else nthreads
    times = []
    t_end = time.time() + seconds
    while True:
        t = time.perf_counter()
        if case.fused:
            oracle.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, nthreads)
        else:
            oracle.rmsnorm_bwd(x, g, dy, rstd, nthreads)
        times.append(time.perf_counter() - t)
        if time.time() >= t_end:
            break
    nbytes = synth.algorithmic_bytes(case.M, case.N, case.dtype, case.with_dres, True)
    return nbytes * len(times) / sum(times) / 1e9, cores, len(times), sum(times)


def oracle_sample_rate(case, kind, seconds, max_call_s=0.15):
    """The fp64 CPU oracle (all host cores) on a bounded row sample of a
    workload: the first rows of the case's inputs, as many as one call can
    take in about max_call_s, called repeatedly for about `seconds`. Returns
    (GB/s of the sample's algorithmic bytes, cores, rows, calls)."""
    import numpy as np
    import torch
    import oracle
    from rmsnorm_backward_bwd_gb300 import synth
    inp = synth.make_inputs(case)
    g = inp["gamma"].to(torch.float64).numpy()

    def rows64(name, r):
        return inp[name][:r].to(torch.float64).numpy() if name in inp else None

    def prepare(r):
        x = rows64("x", r)
        if kind == "fwd":
            return (x,)
        dy = rows64("dy", r)
        if case.fused:
            _, a, rstd = oracle.fused_add_rmsnorm_fwd(x, rows64("residual", r), g,
                                                      np.float32(case.eps), case.dtype)
        else:
            a = x
            _, rstd = oracle.rmsnorm_fwd(x, g, np.float32(case.eps))
        return a, dy, oracle.round_to(rstd, "f32"), rows64("dres", r)

    def call(args):
        if kind == "fwd":
            oracle.rmsnorm_fwd(args[0], g, np.float32(case.eps))
        elif case.fused:
            oracle.fused_add_rmsnorm_bwd(args[0], g, args[1], args[2], args[3])
        else:
            oracle.rmsnorm_bwd(args[0], g, args[1], args[2])

    probe = min(case.M, 64)
    args = prepare(probe)
    t = time.perf_counter()
    call(args)
    per_row = (time.perf_counter() - t) / probe
    rows = int(min(case.M, max(1, max_call_s / max(per_row, 1e-9))))
    args = prepare(rows)
    call(args)
    n, spent = 0, 0.0
    t_end = time.time() + seconds
    while True:
        t = time.perf_counter()
        call(args)
        spent += time.perf_counter() - t
        n += 1
        if time.time() >= t_end:
            break
    if kind == "fwd":
        s = synth.ELEM_BYTES[case.dtype]
        nbytes = rows * case.N * s * 2 + case.N * s + 4 * rows
    else:
        nbytes = synth.algorithmic_bytes(rows, case.N, case.dtype, case.with_dres, True)
    return nbytes * n / spent / 1e9, oracle.max_threads(), rows, n


def workload_runs():
    """The workloads of the benchmark table (besides the headline step): the
    small f32 forward and backward, the edge shapes (plain and fused-add with
    a residual gradient), fused-add 4096 x 4096 with and without it, and the
    16384 x 8192 training shape, plain and fused."""
    from rmsnorm_backward_bwd_gb300 import synth
    runs = [(synth.SMALL_F32, "fwd"), (synth.SMALL_F32, "bwd")]
    runs += [(c, "bwd") for c in synth.edge_cases()]
    runs += [(synth.FUSED_4096, "bwd"), (synth.FUSED_4096_NODRES, "bwd"),
             (synth.LARGE_PLAIN, "bwd"), (synth.LARGE_FUSED, "bwd")]
    return runs


class FwdProblem:
    """Device-resident inputs/outputs of one RMSNorm forward, plus the call."""

    def __init__(self, case, dev):
        import torch
        from rmsnorm_backward_bwd_gb300 import synth
        self.case = case
        inp = synth.make_inputs(case, device=str(dev))
        self.x, self.g = inp["x"], inp["gamma"]
        self.y = torch.empty_like(self.x)
        self.rstd = torch.empty(case.M, dtype=torch.float32, device=dev)
        s = synth.ELEM_BYTES[case.dtype]
        self.bytes = case.M * case.N * s * 2 + case.N * s + 4 * case.M
        torch.cuda.synchronize()

    def call(self):
        import rmsnorm_backward_bwd_gb300 as rn
        rn.rmsnorm_fwd(self.x, self.g, self.case.eps, y=self.y, rstd=self.rstd)


def time_workloads(dev, flush, peak, steps, warmup, ws, cpu_seconds, rank):
    """Every workload run: device us per call (L2 flushed before each call,
    CUDA events), algorithmic GB/s and % of peak, the row-pass kernel time
    and the plan (backward), and the fp64 CPU oracle on the host cores beside
    it (rank 0, single process only)."""
    import numpy as np
    import torch
    from rmsnorm_backward_bwd_gb300 import native
    rows = []
    for case, kind in workload_runs():
        prob = FwdProblem(case, dev) if kind == "fwd" else Problem(case, dev)
        n = max(20, steps // 4)
        cms, _, _ = time_calls(prob, n, warmup, flush, ws)
        t = float(np.mean(cms))
        row = {"workload": ("rmsnorm_fwd %s M=%d N=%d" % (case.dtype, case.M, case.N)
                            if kind == "fwd" else case.name),
               "kind": kind, "us_per_call": round(t * 1e3, 2),
               "GBps": round(prob.bytes / (t * 1e-3) / 1e9, 1),
               "pct_of_peak": round(100 * prob.bytes / (t * 1e-3) / 1e9 / peak, 1),
               "algorithmic_bytes": prob.bytes}
        if kind == "bwd":
            _, kms, _ = time_calls(prob, n, 3, flush, ws, kernel_events=True)
            k = float(np.mean(kms))
            row["row_pass_us"] = round(k * 1e3, 2)
            row["row_pass_GBps"] = round(prob.row_pass_bytes / (k * 1e-3) / 1e9, 1)
        row["plan"] = native.last_plan()
        if rank == 0 and ws == 1 and cpu_seconds > 0:
            rate, cores, srows, calls = oracle_sample_rate(case, kind, cpu_seconds)
            row["cpu_baseline"] = {
                "value": round(rate, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": "%d of %d rows, %d calls (fp64 C oracle, OpenMP)" % (
                    srows, case.M, calls)}
        rows.append(row)
        del prob
        torch.cuda.empty_cache()
    return rows


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, timed as it stands."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1 and rank != 0:
        return
    import numpy as np
    import torch
    import oracle
    from rmsnorm_backward_bwd_gb300 import synth
    case = workload_case(args.workload)
    inp = synth.make_inputs(case)
    x = inp["x"].to(torch.float64).numpy()
    g = inp["gamma"].to(torch.float64).numpy()
    dy = inp["dy"].to(torch.float64).numpy()
    if case.fused:
        _, x, rstd = oracle.fused_add_rmsnorm_fwd(x, inp["residual"].to(torch.float64).numpy(),
                                                  g, np.float32(case.eps), case.dtype)
    else:
        _, rstd = oracle.rmsnorm_fwd(x, g, np.float32(case.eps))
    rstd = oracle.round_to(rstd, "f32")
    dres = inp["dres"].to(torch.float64).numpy() if "dres" in inp else None
    # each step: a bounded sample of the workload's rows (whole problem when
    # it takes under ~0.5 s)
    rows = case.M
    call = (lambda xs, dys, rs, drs: oracle.fused_add_rmsnorm_bwd(xs, g, dys, rs, drs)
            if case.fused else oracle.rmsnorm_bwd(xs, g, dys, rs))
    t = time.perf_counter()
    call(x[:256], dy[:256], rstd[:256], dres[:256] if dres is not None else None)
    per_row = (time.perf_counter() - t) / 256
    rows = int(min(case.M, max(1, 0.5 / max(per_row, 1e-9))))
    xs, dys, rs = x[:rows], dy[:rows], rstd[:rows]
    drs = dres[:rows] if dres is not None else None
    for _ in range(args.warmup):
        call(xs, dys, rs, drs)
    t = time.perf_counter()
    for _ in range(args.steps):
        call(xs, dys, rs, drs)
    dt = (time.perf_counter() - t) / args.steps
    nbytes = synth.algorithmic_bytes(rows, case.N, case.dtype, case.with_dres, True)
    gbs = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case.name, "M": case.M, "N": case.N, "eps": case.eps},
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": "%d of %d rows per step (fp64 C oracle, OpenMP)" % (rows, case.M)},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import numpy as np
    import torch
    from rmsnorm_backward_bwd_gb300 import native

    ws, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or getattr(props, "l2_cache_size", 0) or (128 << 20)
    flush = L2Flush(l2, dev)
    case = workload_case(args.workload)
    prob = Problem(case, dev)
    prob.call()
    torch.cuda.synchronize()
    plan = native.last_plan()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    call_ms, _, wall = time_calls(prob, args.steps, args.warmup, flush, ws, sampler)
    _, kern_ms, _ = time_calls(prob, args.steps, 3, flush, ws, sampler, kernel_events=True)
    clocks = sampler.stop()

    ms = float(np.mean(call_ms))
    ms_max = max_over_ranks(ms, ws)
    kms = max_over_ranks(float(np.mean(kern_ms)), ws)
    value = whole_job_gbs(prob.bytes, ws, ms_max)
    peak, peak_kind = measured_peak()
    achieved = prob.row_pass_bytes / (kms * 1e-3) / 1e9

    e2e_steps = max(3, min(args.steps, 200))
    e2e_ms, h2d, d2h = time_e2e(prob, e2e_steps, 3, ws)
    e2e_ms = max_over_ranks(e2e_ms, ws)

    extra = []
    if not args.no_extra:
        for name in ("plain_4096x32768", "plain_4096x4095", "plain_4096x12290"):
            if name == args.workload:
                continue
            p2 = Problem(workload_case(name), dev)
            n2 = max(20, args.steps // 4)
            cms, _, _ = time_calls(p2, n2, args.warmup, flush, ws)
            _, kms2, _ = time_calls(p2, n2, 3, flush, ws, kernel_events=True)
            t2 = float(np.mean(cms))
            k2 = float(np.mean(kms2))
            extra.append({"workload": p2.case.name, "us_per_call": round(t2 * 1e3, 2),
                          "GBps": round(p2.bytes / (t2 * 1e-3) / 1e9, 1),
                          "pct_of_peak": round(100 * p2.bytes / (t2 * 1e-3) / 1e9 / peak, 1),
                          "row_pass_us": round(k2 * 1e3, 2),
                          "row_pass_GBps": round(p2.row_pass_bytes / (k2 * 1e-3) / 1e9, 1),
                          "plan": native.last_plan()})
            del p2
            torch.cuda.empty_cache()
        from rmsnorm_backward_bwd_gb300 import synth as _synth
        for ln_case in (_synth.LN_4096, _synth.LN_LARGE, _synth.LN_UNALIGNED):
            p3 = LnProblem(ln_case, dev)
            n3 = max(20, args.steps // 4)
            cms, _, _ = time_calls(p3, n3, args.warmup, flush, ws)
            _, kms3, _ = time_calls(p3, n3, 3, flush, ws, kernel_events=True)
            t3, k3 = float(np.mean(cms)), float(np.mean(kms3))
            extra.append({"workload": p3.case.name + " (dgamma + dbeta)",
                          "us_per_call": round(t3 * 1e3, 2),
                          "GBps": round(p3.bytes / (t3 * 1e-3) / 1e9, 1),
                          "pct_of_peak": round(100 * p3.bytes / (t3 * 1e-3) / 1e9 / peak, 1),
                          "row_pass_us": round(k3 * 1e3, 2),
                          "row_pass_GBps": round(p3.row_pass_bytes / (k3 * 1e-3) / 1e9, 1),
                          "plan": native.last_plan()})
            del p3
            torch.cuda.empty_cache()

    steady = []
    if not args.no_extra:
        for name in ("plain_4096", "fused_4096_nodres", "fused_4096", "plain_4096x4095",
                     "plain_16384x8192"):
            c4 = workload_case(name)
            sms, R, ncalls, splan = time_steady(c4, dev, args.steps, ws, l2)
            b4 = synth_bytes(c4)
            steady.append({"workload": c4.name, "us_per_call": round(sms * 1e3, 2),
                           "GBps": round(b4 / (sms * 1e-3) / 1e9, 1),
                           "pct_of_peak": round(100 * b4 / (sms * 1e-3) / 1e9 / peak, 1),
                           "input_sets": R, "calls_timed": ncalls, "plan": splan})

    workloads = []
    if not args.no_extra:
        workloads = time_workloads(dev, flush, peak, args.steps, args.warmup, ws,
                                   0.0 if args.no_cpu else args.workload_cpu_seconds, rank)

    forward = []
    pages_table = []
    if not args.no_extra:
        forward = time_forwards(dev, flush, max(20, args.steps // 10), args.warmup, peak)
        pages_table = autograd_pages_table(dev)

    autograd = []
    if not args.no_extra:
        for name in ("plain_4096", "fused_4096", "layernorm_4096"):
            c2 = workload_case(name)
            nbytes = synth_bytes(c2)
            row = {"workload": c2.name}
            grads = {}
            for impl in ("ours", "torch_eager"):
                g = autograd_problem(c2, dev, impl)
                grads[impl] = [t.float() for t in torch.autograd.grad(*g, retain_graph=True)]
                n3 = max(20, args.steps // 4)
                t = time_autograd(g, n3, args.warmup, flush)
                tq = time_autograd(g, n3, args.warmup, flush, queued=True)
                row[impl + "_us"] = round(t * 1e3, 2)
                row[impl + "_GBps"] = round(nbytes / (t * 1e-3) / 1e9, 1)
                row[impl + "_device_us"] = round(tq * 1e3, 2)
                row[impl + "_device_GBps"] = round(nbytes / (tq * 1e-3) / 1e9, 1)
                del g
                torch.cuda.empty_cache()
            # gradients compared before timing is reported (largest difference
            # relative to the tensor's largest magnitude, over x/residual/weight)
            row["max_rel_diff_vs_torch_eager"] = float("%.3g" % max(
                float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))
                for a, b in zip(grads["ours"], grads["torch_eager"])))
            del grads
            row["speedup_vs_torch_eager"] = round(row["torch_eager_us"] / row["ours_us"], 2)
            row["device_speedup_vs_torch_eager"] = round(
                row["torch_eager_device_us"] / row["ours_device_us"], 2)
            autograd.append(row)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        rate, cores, n, secs = oracle_rate(case, args.cpu_seconds)
        cpu = {"value": round(rate, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": "full %dx%d problem, %d calls in %.1f s (fp64 C oracle, OpenMP)" % (
                   case.M, case.N, n, secs)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
            "us_per_call": round(ms_max * 1e3, 2),
            "pct_of_peak": round(100 * value / ws / peak, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": case.dtype, "data": "synthetic",
            "config": {"workload": case.name, "M": case.M, "N": case.N, "eps": case.eps,
                       "step": "one backward call: row pass + weight-gradient reduction + cast",
                       "l2": "flushed before every step: write %d MiB, then read %d MiB "
                             "(2x L2 each)" % (flush.mib, flush.mib),
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic(args.workload), "kernel": row_pass_kernel(plan),
                         "peak_source": peak_kind,
                         "algorithmic_bytes_per_launch": prob.row_pass_bytes,
                         "us_per_launch": round(kms * 1e3, 2)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(whole_job_gbs(prob.bytes, ws, e2e_ms), 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": launches_per_call(plan) * args.steps,
            "clocks": clocks,
            "plan": plan,
            "workloads": workloads,
            "extra": extra,
            "steady": steady,
            "autograd": autograd,
            "forward": forward,
            "autograd_pages_shapes": pages_table,
        }
        # every backward workload's device time and % of peak also as flat top-level keys, so
        # that a record keeping only scalars keeps them too
        for w in workloads or []:
            if w.get("kind") != "bwd":
                continue
            slug = re.sub(r"[^0-9a-z]+", "_", w["workload"].lower().replace(" m=", " ")
                          .replace(" n=", "x")).strip("_")
            line["us_per_call__" + slug] = w["us_per_call"]
            line["pct_of_peak__" + slug] = w["pct_of_peak"]
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="plain_4096",
                    choices=["plain_4096", "fused_4096", "fused_4096_nodres", "plain_16384x8192",
                             "fused_16384x8192", "plain_4096x32768", "plain_4096x4095",
                             "plain_4096x12290"])
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload-cpu-seconds", type=float, default=1.0,
                    help="oracle time per workload of the workload table")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
        return
    import __graft_entry__
    __graft_entry__.build()
    run_ours(args)


if __name__ == "__main__":
    main()
