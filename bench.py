"""Benchmark of the gated delta rule library on one node.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]
                    [--workload decode-L1|decode-L4|decode-L1-kmajor|decode-L4-kmajor|
                                ragged-prefill|long-prefill-<rule>|gdn2|gdn2-gates|gated-perkey]
                    [--no-extra]

A step is one call of the library on one batch of the workload (the decode
workload: 256 requests of L tokens, Hq=16, Hv=32, dk=dv=128, fp16
activations, an fp32 state slab [1024, 32, 128, 128] updated in place at
permuted slot ids, raw gate and beta through the fused arm).  Inputs are
seeded synthetic draws (workloads.py) resident in HBM.  Timing: W untimed
warm-up steps, then K steps between a barrier + synchronize on both sides,
CUDA events on the launching stream; the touched state (512 MiB) exceeds
the 129 MB L2 every step, so no extra flush is needed.  Rank 0 prints one
JSON line.  With N > 1 each rank runs its own independent batch (weak
scaling: the work partitions over requests; no collective on the data path).

--impl reference times the CPU oracle (the only other implementation there
is) on the host cores on bounded samples of the same workload.
"""
import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "tokens/s per GDN layer (decode, prefill) and % of HBM / tensor-core roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILES = os.path.join(ROOT, "profiles")
ESZ = {torch.float16: 2, torch.float32: 4, torch.int32: 4}
CHUNK = 64


# ------------------------------------------------------------------ workloads
def make_workload(name, seed_offset=0, shrink=1):
    """The named workload; ``shrink`` > 1 divides its request count or
    sequence length (a smaller case of the same kernel, for profiling)."""
    if name.startswith("decode-L"):
        km = name.endswith("-kmajor")
        L = int(name[len("decode-L"):].split("-")[0])
        p = workloads.decode(L, seed=2 + seed_offset, B=256 // shrink, num_slots=1024 // shrink)
        if km:  # the same slab stored key-major, [rows, Hv, dk, dv]
            p = dict(p, state_kmajor=True, initial_state=p["initial_state"].transpose(2, 3).contiguous())
        return p, "recurrent"
    if name == "ragged-prefill":
        return workloads.ragged_prefill(seed=3 + seed_offset, total=16384 // shrink,
                                        max_len=4096 // shrink), "chunked"
    if name.startswith("long-prefill-"):
        return workloads.long_prefill(name[len("long-prefill-"):], seed=4 + seed_offset,
                                      S=8192 // shrink), "chunked"
    if name == "gdn2":
        return workloads.gdn2(seed=5 + seed_offset, S=4096 // shrink), "chunked"
    if name == "gated-perkey":  # the gated rule with per-key decay (GLA-style gating)
        return workloads.gated_perkey(seed=6 + seed_offset, S=4096 // shrink), "chunked"
    if name == "gdn2-gates":  # erase gate as its own input beside a scalar beta, write gate passed in
        return workloads.gdn2(seed=5 + seed_offset, S=4096 // shrink, erase="input", write_gate="input"), "chunked"
    raise SystemExit("unknown workload " + name)


def _nbytes(t):
    return 0 if t is None else t.numel() * ESZ.get(t.dtype, t.element_size())


def algorithmic_bytes(p):
    """Each input read once, each output written once, the touched state rows
    read (if an initial state is given) and written once."""
    b = sum(_nbytes(p.get(k)) for k in ("q", "k", "v", "decay", "gate_bias", "gate_scale", "beta",
                                         "erase_gate", "write_gate", "cu_seqlens", "slot_ids"))
    b += _nbytes(p["v"])  # o, same shape and dtype as v
    tile = p["batch"] * p["hv"] * p["dv"] * p["dk"] * 4
    b += tile * (2 if p.get("initial_state") is not None else 1)
    return b


def algorithmic_flops(p, C=CHUNK):
    """Dense tile counts of the chunked form per (token, value head):
    6 dk dv + 2C(3dk + 2dv) with retrieval, 4 dk dv + 2C(dk + dv) without."""
    dk, dv = p["dk"], p["dv"]
    if p["rule"] in ("delta", "gated_delta", "gdn2"):
        per = 6 * dk * dv + 2 * C * (3 * dk + 2 * dv)
    else:
        per = 4 * dk * dv + 2 * C * (dk + dv)
    return per * p["total_tokens"] * p["hv"]


def tokens(p):
    return sum(t1 - t0 for t0, t1 in workloads.token_ranges(p))


# ------------------------------------------------------------------ clocks
class NvmlClocks:
    """Samples the SM clock and the clock event reasons through NVML (ctypes,
    read-only queries) every millisecond in a thread, so that even a timed
    region of a few milliseconds holds several samples."""
    # nvmlClocksEventReason* bits of the NVML API
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}

    def __init__(self, device_index=0):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML handle for " + uuid)
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples = []
        self.run = False

    def _one(self):
        ct = self.ct
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(mhz)) != 0:  # NVML_CLOCK_SM
            return None
        if self.reasons_fn(self.dev, ct.byref(rs)) != 0:
            rs.value = 0
        return mhz.value, rs.value

    def _loop(self):
        while self.run:
            x = self._one()
            if x:
                self.samples.append(x)
            time.sleep(0.001)

    def start(self):
        self.samples = []
        self.run = True
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 1.0:
            time.sleep(0.0005)

    def stop(self):
        self.run = False
        self.thread.join(timeout=2)
        mx = self.ct.c_uint()
        smax = mx.value if self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, self.ct.byref(mx)) == 0 else None
        sm = [m for m, _ in self.samples]
        reasons = sorted(nm for nm, bit in self.REASONS.items() if any(r & bit for _, r in self.samples))
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(sm), "source": "nvml, 1 ms"}


class SmiClocks:
    """The same from nvidia-smi (20 ms samples), where NVML cannot be loaded."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.lines = []
        self.skip = 0
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                    "-lms", "20"] + sel

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # nvidia-smi takes a moment to start: wait for its first sample so that
        # the samples taken afterwards fall inside the timed region
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.skip = len(self.lines)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines[self.skip:] or self.lines[-1:]
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 20 ms"}




def clock_sampler(device_index=0):
    try:
        return NvmlClocks(device_index)
    except Exception:
        return SmiClocks(device_index)


# ------------------------------------------------------------------ device runs
def to_dev(p, dev):
    d = dict(p)
    for k in ("q", "k", "v", "decay", "gate_bias", "gate_scale", "beta", "erase_gate", "write_gate",
              "cu_seqlens", "slot_ids", "initial_state"):
        if p.get(k) is not None:
            d[k] = p[k].to(dev).contiguous()
    return d


def build_problem(api, p, d, o, fin):
    q, k, v = d["q"], d["k"], d["v"]
    if p.get("seq_len"):
        B, S = p["batch"], p["seq_len"]
        q = q.view(B, S, p["hq"], p["dk"])
        k = k.view(B, S, p["hq"], p["dk"])
        v = v.view(B, S, p["hv"], p["dv"])
        o = o.view(B, S, p["hv"], p["dv"])
    init = fin if p.get("slot_ids") is not None else d.get("initial_state")
    return api.make_problem(q=q, k=k, v=v, o=o, final_state=fin, rule=p["rule"],
                            decay=d.get("decay"), beta=d.get("beta"), gate_bias=d.get("gate_bias"),
                            gate_scale=d.get("gate_scale"), cu_seqlens=d.get("cu_seqlens"),
                            slot_ids=d.get("slot_ids"), initial_state=init, batch=p["batch"],
                            scale=p.get("scale", 0.0), l2norm_q=p.get("l2norm_q", False),
                            l2norm_k=p.get("l2norm_k", False),
                            beta_sigmoid=p.get("beta_sigmoid", False),
                            decay_per_key=p.get("decay_per_key", False),
                            erase_gate=d.get("erase_gate"), write_gate=d.get("write_gate"),
                            state_kmajor=p.get("state_kmajor", False))


def launch(api, prob, path, stream):
    if path == "recurrent":
        api.gdn_recurrent_step(prob, stream=stream)
    else:
        api.gdn_chunked_prefill(prob, chunk_size=CHUNK, workspace=prob._ws_buf, stream=stream)


def prepare(api, p, path, dev):
    d = to_dev(p, dev)
    o = torch.empty_like(d["v"])
    rows = p.get("num_slots") or p["batch"]
    if p.get("slot_ids") is not None:
        fin = d["initial_state"]  # the slab, updated in place
    else:
        shape = (rows, p["hv"], p["dk"], p["dv"]) if p.get("state_kmajor") else (rows, p["hv"], p["dv"], p["dk"])
        fin = torch.empty(*shape, dtype=torch.float32, device=dev)
    prob = build_problem(api, p, d, o, fin)
    prob._ws_buf = None
    if path == "chunked":
        n = api.gdn_chunked_prefill_workspace_size(prob, CHUNK)
        prob._ws_buf = torch.empty(max(n, 1), dtype=torch.uint8, device=dev) if n else None
    return d, o, fin, prob


def time_device(api, prob, path, steps, warmup, stream, barrier):
    for _ in range(warmup):
        launch(api, prob, path, stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        launch(api, prob, path, stream)
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    total_ms = t0.elapsed_time(t1)
    per_launch = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return total_ms, per_launch


E2E_REPEATS = 3  # timed end-to-end regions per measurement (their median is reported)


def time_e2e(api, p, d, prob, path, steps, warmup, stream, dev):
    """Every step: pinned host -> device copies of the step's inputs, the call,
    and a device -> host copy of the output.  Steps run through two sets of
    device input and output buffers, with the copies on their own streams, so
    the input copies of one step overlap the call of the step before and its
    output copy (the other direction) the input copies of the step after; the
    state (slab or final state) and the workspace are shared and the calls run
    in order on ``stream``.  The timed region spans the first input copy to the
    last output copy; it runs ``E2E_REPEATS`` times and the median is returned
    (the host link is shared, and a transient on it can halve one region)."""
    names = [k for k in ("q", "k", "v", "decay", "beta", "erase_gate", "write_gate", "cu_seqlens", "slot_ids")
             if p.get(k) is not None]
    host = {k: p[k].contiguous().pin_memory() for k in names}
    o_dev = prob._keep[3]
    fin = prob._keep[4]
    d2 = dict(d)
    for k in names:
        d2[k] = torch.empty_like(d[k])
    o2 = torch.empty_like(o_dev)
    prob2 = build_problem(api, p, d2, o2, fin)
    prob2._ws_buf = prob._ws_buf
    sets = [(d, prob, o_dev), (d2, prob2, o2)]
    o_host = [torch.empty(p["v"].shape, dtype=p["v"].dtype).pin_memory() for _ in range(2)]
    h2d = sum(_nbytes(host[k]) for k in names)
    d2h = _nbytes(o_host[0])
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def one(i):
        b = i & 1
        dd, pr, od = sets[b]
        if i >= 2:
            cin.wait_event(ev_done[b])  # the call of step i - 2 has read this input set
        with torch.cuda.stream(cin):
            for k in names:
                dd[k].copy_(host[k], non_blocking=True)
        ev_in[b].record(cin)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # the output of step i - 2 has been copied out
        launch(api, pr, path, stream)
        ev_done[b].record(stream)
        cout.wait_event(ev_done[b])
        with torch.cuda.stream(cout):
            o_host[b].copy_(od.view(o_host[b].shape), non_blocking=True)
        ev_out[b].record(cout)

    def run(n):
        start = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        cin.wait_event(start)
        for i in range(n):
            one(i)
        for b in range(min(n, 2)):
            stream.wait_event(ev_out[b])
        end = torch.cuda.Event(enable_timing=True)
        end.record(stream)
        return start, end

    run(warmup)
    torch.cuda.synchronize()
    times = []
    for _ in range(E2E_REPEATS):
        t0, t1 = run(steps)
        torch.cuda.synchronize()
        times.append(t0.elapsed_time(t1))
    return statistics.median(times), h2d, d2h


def kernel_name(p, path):
    """The kernel the library dispatches for this workload (mirrors the host
    dispatch in the CUDA sources)."""
    def token_serial():
        # average request length above four staged token blocks (of 8): the long-request kernel
        L = p.get("seq_len") or p["total_tokens"] // max(p["batch"], 1)
        if L > 32:
            return "recurrent_long_kernel<%d>" % p["dk"]
        return "recurrent_pipe_kernel<%d,%s>" % (p["dk"], "true" if p.get("state_kmajor") else "false")
    if path == "recurrent":
        return token_serial()
    per_key = p.get("decay_per_key") and p["rule"] in ("gated", "gated_delta", "gdn2")
    # fp32 activations go through fp16 copies, fp16 per-key gate rows through fp32 copies
    tc_shape = p["dk"] == 128 and p["dv"] == 128
    if tc_shape and (p["rule"] == "gdn2" or (per_key and p["rule"] in ("gated", "gated_delta"))):
        return "chunk_prepare_perkey_kernel<%d>+chunk_chain_kernel<2>" % int(p["rule"] == "gdn2")
    if per_key:
        return token_serial()
    if tc_shape and p["rule"] != "gdn2":
        retr = p["rule"] in ("delta", "gated_delta")
        return "chunk_prepare_kernel<%d>+chunk_chain_kernel<%d>" % (
            int(retr), {"linear": 0, "gated": 1}.get(p["rule"], 2))
    return "chunked_mma_kernel<%d,%s>" % (p["dk"], "true" if p["rule"] == "gdn2" else "false")


def launches_per_call(p, path):
    """Kernels one library call launches: the tensor-core prefill runs the
    chunk-offset scan and the per-chunk operand pass (with the triangular
    solves for the delta rules) before the chain."""
    k = kernel_name(p, path)
    if "chunk_chain_kernel" not in k:
        return 1
    n = 3 + (3 if p["act_dtype"] == "f32" else 0)  # + the fp16 copies of q, k, v
    if "perkey" in k:  # + the fp32 copies of fp16 per-key gate rows
        if p.get("decay_per_key") and p["decay"].dtype == torch.float16:
            n += 1
        if p["rule"] == "gdn2" and p.get("erase_gate") is None and p["beta"].dtype == torch.float16:
            n += 1
    return n


def kernel_source_digest(path, kernel=""):
    """SHA-256 prefix of the sources the dispatched kernels are built from."""
    if kernel.startswith("recurrent"):
        names = ["recurrent.cu"]
    elif kernel.startswith(("chunk_chain", "chunk_prepare")):
        names = ["chunked_tc.cu", "chunk_image.cuh"] + (
            ["chunked_tc_perkey.cu"] if "perkey" in kernel else [])
    else:
        names = ["chunked.cu"]
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "gated_delta_rule_gate_gb300", "csrc", name)) as fh:
            text = fh.read()
        # the code only: comments and blank lines do not change a kernel
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload, path, kernel=""):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; None otherwise."""
    f = os.path.join(PROFILES, "traffic.json")
    try:
        with open(f) as fh:
            data = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = data.get(workload)
    if not ent or ent.get("source_sha256_16") != kernel_source_digest(path, kernel):
        return None
    return ent.get("dram_bytes_per_launch")


def peaks():
    try:
        with open(PEAKS_FILE) as fh:
            pk = json.load(fh)
        return pk["hbm_gbs"], pk["bf16_tflops"], pk.get("bf16_tflops_sustained"), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ CPU oracle
def oracle_rate(p, budget_s, threads, max_requests=None, real="f64"):
    """Oracle tokens/s on a bounded sample of the workload's requests (all
    value heads of each sampled request).  Grows the sample until one timed
    pass takes >= budget_s seconds (or covers every request).  ``real``: the
    double build (the definition) or its float instantiation."""
    import oracle
    ranges = workloads.token_ranges(p)
    order = [b for b in range(p["batch"]) if ranges[b][1] > ranges[b][0]]
    n = 1
    while True:
        sample = order[:n]
        t = time.perf_counter()
        oracle.run_problem(p, requests=sample, threads=threads, real=real)
        dt = time.perf_counter() - t
        toks = sum(ranges[b][1] - ranges[b][0] for b in sample)
        if dt >= budget_s or n >= len(order) or (max_requests and n >= max_requests):
            return toks / dt, sample, toks, dt
        n = min(len(order), max(n + 1, int(n * max(2.0, 1.2 * budget_s / max(dt, 1e-3)))))


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ arms
def run_reference(args, rank):
    if rank != 0:
        return
    p, path = make_workload(args.workload, shrink=args.shrink)
    cores = cpu_cores()
    import oracle
    ranges = workloads.token_ranges(p)
    order = [b for b in range(p["batch"]) if ranges[b][1] > ranges[b][0]]
    # size one step: enough requests for ~0.05 s, capped so K + W steps stay in minutes
    _, sample, toks, dt = oracle_rate(p, 0.05, cores)
    per_step_s = dt
    budget = 150.0
    if (args.steps + args.warmup) * per_step_s > budget and len(sample) > 1:
        keep = max(1, int(len(sample) * budget / ((args.steps + args.warmup) * per_step_s)))
        sample = sample[:keep]
    toks = sum(ranges[b][1] - ranges[b][0] for b in sample)
    for _ in range(args.warmup):
        oracle.run_problem(p, requests=sample, threads=cores)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.run_problem(p, requests=sample, threads=cores)
        times.append(time.perf_counter() - t)
    total = sum(times)
    value = toks * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(p, args, note="oracle on %d of %d requests per step" %
                                  (len(sample), p["batch"])),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "%d requests x %d value heads (%d tokens) per step" %
                                   (len(sample), p["hv"], toks)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(p, args, note=None):
    cfg = {"workload": args.workload, "batch": p["batch"], "total_tokens": p["total_tokens"],
           "seq_len": p.get("seq_len") or None, "Hq": p["hq"], "Hv": p["hv"], "dk": p["dk"],
           "dv": p["dv"], "rule": p["rule"], "act_dtype": p["act_dtype"],
           "state": "fp32 " + ("K-major" if p.get("state_kmajor") else "V-major"), "parallelism": "replicas" if args.gpus > 1 else "single-gpu",
           "l2_policy": "inputs larger than L2 (touched state > 129 MB)"}
    if p.get("num_slots") and p.get("slot_ids") is not None:
        cfg["slab_rows"] = p["num_slots"]
    if note:
        cfg["note"] = note
    return cfg


def roofline(p, path, workload, kern_ms):
    """Algorithmic bytes (and flops) per launch over the mean launch time,
    against the measured peaks."""
    hbm, tc, tc_s, src = peaks()
    ab = algorithmic_bytes(p)
    achieved = ab / (kern_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": ncu_traffic(workload, path, kernel_name(p, path)), "kernel": kernel_name(p, path),
            "algorithmic_bytes_per_launch": ab, "peak_source": src + " (MEASURED_PEAKS.json hbm_gbs)"}
    if path == "chunked":
        af = algorithmic_flops(p)
        roof["tensor_achieved_tflops"] = af / (kern_ms * 1e-3) / 1e12
        roof["tensor_frac"] = roof["tensor_achieved_tflops"] / tc
        roof["algorithmic_flops_per_launch"] = af
    return roof


def cpu_baseline(p, budget_s, single_thread_budget=None):
    """The oracle on the host cores: the double build on every core; with
    ``single_thread_budget`` also on one core, and its float instantiation on
    every core and on one."""
    cores = cpu_cores()
    rate, sample, stoks, sdt = oracle_rate(p, budget_s, cores)
    fmt = "%d of %d requests, all %d value heads (%d tokens, %.1f s), %s"
    out = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": fmt % (len(sample), p["batch"], p["hv"], stoks, sdt, "fp64")}
    if single_thread_budget:
        r1, s1, t1, d1 = oracle_rate(p, single_thread_budget, 1)
        out["single_thread"] = {"value": r1, "unit": "tokens/s", "cores": 1,
                                "sample": fmt % (len(s1), p["batch"], p["hv"], t1, d1, "fp64")}
        rf, sf, tf, df = oracle_rate(p, single_thread_budget, cores, real="f32")
        rf1, sf1, tf1, df1 = oracle_rate(p, single_thread_budget, 1, real="f32")
        out["float32"] = {"value": rf, "unit": "tokens/s", "cores": cores,
                          "sample": fmt % (len(sf), p["batch"], p["hv"], tf, df, "fp32 instantiation")}
        out["float32_single_thread"] = {"value": rf1, "unit": "tokens/s", "cores": 1,
                                        "sample": fmt % (len(sf1), p["batch"], p["hv"], tf1, df1,
                                                         "fp32 instantiation")}
    return out


def extra_workloads(api, dev, stream, names, with_cpu=True, region_s=0.2, warmup=5):
    """Each other workload measured like the headline one: device time of a
    timed region of about region_s seconds with clocks sampled inside it, its
    roofline, an end-to-end figure with host copies, and the CPU oracle on a
    bounded sample of it."""
    out = {}
    for name in names:
        p, path = make_workload(name)
        try:
            d, o, fin, prob = prepare(api, p, path, dev)
        except Exception as e:  # an unsupported configuration is reported, not hidden
            out[name] = {"error": str(e)[:200]}
            continue
        est, _ = time_device(api, prob, path, 5, warmup, stream, lambda: None)
        steps = int(min(2000, max(20, math.ceil(region_s * 1e3 / max(est / 5, 1e-3)))))
        clocks = clock_sampler(dev.index or 0)
        clocks.start()
        total, per = time_device(api, prob, path, steps, 3, stream, lambda: None)
        clk = clocks.stop()
        ms = total / steps
        toks = tokens(p)
        ent = {"tokens_per_s": toks / (ms * 1e-3), "ms_per_call": ms, "steps": steps, "path": path,
               "roofline": roofline(p, path, name, statistics.fmean(per)), "clocks": clk,
               "gpu_launches": steps * launches_per_call(p, path)}
        e2e_ms, h2d, d2h = time_e2e(api, p, d, prob, path, 10, 3, stream, dev)
        ent["e2e"] = {"value": toks / (e2e_ms / 10 * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "repeats": E2E_REPEATS}
        if with_cpu:
            ent["cpu_baseline"] = cpu_baseline(p, 1.0)
        out[name] = ent
        del d, o, fin, prob
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--workload", default="decode-L1")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end timing")
    ap.add_argument("--shrink", type=int, default=1,
                    help="divide the workload's requests or length (profiling runs)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "gdn" else "gloo")
    if args.impl == "reference":
        run_reference(args, rank)
        if dist:
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import gated_delta_rule_gate_gb300 as pkg
    from gated_delta_rule_gate_gb300 import api
    pkg.load()

    def barrier():
        if dist:
            dist.barrier()

    p, path = make_workload(args.workload, seed_offset=100 * rank, shrink=args.shrink)
    d, o, fin, prob = prepare(api, p, path, dev)
    stream = torch.cuda.current_stream(dev)

    clocks = clock_sampler(local)
    clocks.start()
    total_ms, per_launch = time_device(api, prob, path, args.steps, args.warmup, stream, barrier)
    clk = clocks.stop()

    toks = tokens(p)
    if dist:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms = total_ms / args.steps
    value = toks * world / (ms * 1e-3)

    if args.no_e2e:
        e2e = None
    else:
        e2e_steps = max(1, min(args.steps, 50))
        e2e_ms, h2d, d2h = time_e2e(api, p, d, prob, path, e2e_steps, 3, stream, dev)
        e2e = {"value": toks * world / (e2e_ms / e2e_steps * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "repeats": E2E_REPEATS}

    roof = roofline(p, path, args.workload, statistics.fmean(per_launch))

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, workloads.py)", "config": workload_config(p, args),
        "roofline": roof, "clocks": clk,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_call(p, path),
    }
    if rank == 0:
        if args.shrink > 1:
            line["config"]["shrink"] = args.shrink
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(p, 3.0, single_thread_budget=2.0)
    if rank == 0:
        if not args.no_extra and world == 1:
            names = [n for n in ("decode-L1", "decode-L4", "decode-L1-kmajor", "decode-L4-kmajor",
                                 "ragged-prefill", "long-prefill-linear", "long-prefill-gated",
                                 "long-prefill-delta", "long-prefill-gated_delta", "gdn2", "gdn2-gates",
                                 "gated-perkey")
                     if n != args.workload]
            del d, o, fin, prob
            torch.cuda.empty_cache()
            line["other_workloads"] = extra_workloads(api, dev, stream, names, with_cpu=not args.no_cpu)
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
