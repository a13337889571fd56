#!/usr/bin/env python3
"""Throughput of the DSA hot path (fused Lightning Indexer top-K + Sparse Flash Attention).

One step = one pass of the whole path over one batch: li_topk then sfa_decode (sfa_prefill for
the prefill workload), launched through the C ABI.  Default workload: decode, 32 sequences x 1
token at 32768 context, 64x128 index heads, top-2048, 128 attention heads over the 576/512 MLA
latent cache (bf16).

Prints ONE JSON line (rank 0):
  value      tokens/s over all ranks, inputs resident in HBM (max over ranks of the timed region)
  e2e        the same through host buffers: per step, the step's query-side inputs are copied
             host->device from pinned memory and the outputs device->host, inside the timed region
  roofline   the dominant kernel: algorithmic bytes (decode; flops for prefill) per launch / its
             median CUDA-event duration, timed alone over 50+ launches, vs the measured HBM
             copy bandwidth (bf16 tensor throughput); traffic from the committed ncu summary
  kernels    the same figures for both kernels
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample of the same workload
Multi-GPU (torchrun): every rank runs its own independently seeded batch (weak scaling, no
collective on the data path).  ``--impl reference`` times the CPU oracle instead.
"""
import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LI+SFA decode tokens/sec at 32k ctx; achieved HBM GB/s vs ~8 TB/s peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_32k")
    ap.add_argument("--baseline-seconds", type=float, default=15.0,
                    help="CPU oracle sample budget for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--query-sets", type=int, default=4,
                    help="independently drawn query sets the steps rotate over")
    ap.add_argument("--kernel-reps", type=int, default=50,
                    help="launches per kernel in the per-kernel timing passes (at least 50)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps eagerly instead of replaying a CUDA graph of them")
    return ap.parse_args()


# ----------------------------------------------------------------------------- bytes / flops

def algorithmic(wl, cnt_total):
    """Per-step algorithmic work: key pages every token's visible range touches (read once per
    sequence), gathered latent rows (one 1152-byte row per selected index), FLOPs."""
    P = wl.page_size
    elt = 2 if wl.li_dtype == "bf16" else 1
    pages = sum(math.ceil(L / P) for L in wl.seq_lens)
    # key scales: one fp32 per row (fp8), one E8M0 byte per 32 elements (mxfp8)
    sc = {"bf16": 0, "fp8": 4, "mxfp8": wl.d_I // 32}[wl.li_dtype]
    k_bytes = pages * P * (wl.d_I * elt + sc)
    gather_bytes = cnt_total * (608 if wl.kv_dtype == "fp8" else wl.d_qk * 2)  # bytes per row
    li_flop = 0
    for L, n in zip(wl.seq_lens, wl.n_new):
        li_flop += sum(2 * (L - n + i + 1) * wl.H_I * wl.d_I for i in range(n))
    sfa_flop = cnt_total * wl.H * (wl.d_qk + wl.d_v) * 2
    return {"k_bytes": k_bytes, "gather_bytes": gather_bytes, "metric_bytes": k_bytes + gather_bytes,
            "li_flop": li_flop, "sfa_flop": sfa_flop}


# ----------------------------------------------------------------------------- clocks (NVML)

class ClockSampler:
    """Polls SM clock and clock-event reasons through NVML (ctypes) while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting"}

    def __init__(self, pci_bus_id):
        self.ok = False
        self.samples, self.reasons = [], 0
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if pci_bus_id is None or self.nv.nvmlDeviceGetHandleByPciBusId_v2(
                    pci_bus_id.encode(), ctypes.byref(self.h)) != 0:
                if self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0:
                    return
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.ok = True
        except Exception:
            self.ok = False

    def _poll(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(r)) == 0:
                self.reasons |= r.value
            self._first.set()
            time.sleep(0.0005)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._first = threading.Event()
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
            self._first.wait(1.0)  # polling has begun before the caller's timed region starts
        self.n_start = len(self.samples)
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def mark(self):
        """Record how many samples the first window (the timed region) holds."""
        self.n_first = len(self.samples) - self.n_start

    def summary(self):
        used = self.samples[getattr(self, "n_start", 0):]  # from the start of the caller's window
        if not self.ok or not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml_unavailable"]}
        out = {"sm_mhz": statistics.median(used), "sm_max_mhz": self.max_mhz,
               "samples": len(used),
               "reasons": [n for b, n in self.REASONS.items() if self.reasons & b]}
        if getattr(self, "n_first", None) is not None:
            out["samples_timed_region"] = self.n_first
            out["window"] = "timed region + per-kernel passes"
        return out


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


def committed_traffic(workload, kernel="li_topk"):
    """Per-launch DRAM bytes of a kernel at a workload from the committed ncu summary, if the
    kernel's source is unchanged since it was taken (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload if kernel == "li_topk" else "%s/%s" % (workload, kernel))
    if not e:
        return None
    src = os.path.join(ROOT, "dsa_sparse_attention_li_gb300", "csrc", e["source"])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return e["dram_bytes_per_launch"] if sha == e["source_sha256_16"] else None


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


# ----------------------------------------------------------------------------- CPU oracle timing

def oracle_sample_rate(inp_cpu, budget_s, tokens_per_call=None):
    """Tokens/s of the oracle (indexer top-K + attention on its own selection) over a bounded
    sample of the workload's tokens."""
    import numpy as np
    import oracle
    wl = inp_cpu["wl"]
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    n = tokens_per_call or min(wl.n_q, max(1, cores))
    rng = np.random.default_rng(5)
    done, t_total, calls = 0, 0.0, 0
    while t_total < budget_s:
        toks = sorted(rng.choice(wl.n_q, size=n, replace=False).tolist())
        t0 = time.perf_counter()
        idx, _, _ = oracle.li_topk(inp_cpu, toks)
        oracle.sfa(inp_cpu, idx, toks)
        t_total += time.perf_counter() - t0
        done += n
        calls += 1
    return done / t_total, cores, "%d calls x %d tokens of %s (%.1f s)" % (calls, n, wl.name, t_total)


def run_reference(args):
    """The CPU oracle as it stands, on this host's cores: each step runs the whole path (indexer
    full-sort top-K, then attention on that selection) for a bounded sample of the workload's
    query tokens, sized so that warm-up + timed steps take about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import dsa_inputs as di
    import oracle
    wl = di.preset(args.workload)
    inp_cpu = di.generate(wl, device="cpu")
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    rng = np.random.default_rng(5)

    def call(n):
        toks = sorted(rng.choice(wl.n_q, size=n, replace=False).tolist())
        t0 = time.perf_counter()
        idx, _, _ = oracle.li_topk(inp_cpu, toks)
        oracle.sfa(inp_cpu, idx, toks)
        return time.perf_counter() - t0

    t_one = call(1)  # calibration (part of the warm-up)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(wl.n_q, cores * max(1, math.floor(budget / max(t_one, 1e-6))))))
    for _ in range(max(0, args.warmup - 1)):
        call(n)
    times = [call(n) for _ in range(max(1, args.steps))]
    value = n * len(times) / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * statistics.mean(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": wl.describe(),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "each step: the fp64 oracle (indexer full-sort top-K + "
                                       "direct softmax attention) on %d of the %d query tokens"
                                       % (n, wl.n_q)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def _median_launch_ms(lib, launch, arg_sets, sp, stream, n):
    """Median CUDA-event duration of ``n`` launches of one entry point alone (rotating over the
    argument sets), each bracketed by its own events on the launching stream."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            ev[i][0].record(stream)
            if launch(ctypes.byref(arg_sets[i % len(arg_sets)]), sp):
                raise RuntimeError("launch failed: " + lib.dsa_last_error().decode())
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)


def run_ours(args):
    import torch
    import dsa_inputs as di
    import dsa_sparse_attention_li_gb300 as dsa

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    lib = dsa.load()

    wl = di.preset(args.workload)
    if world > 1:
        wl = di.Workload(**{**wl.__dict__, "seed": wl.seed + 100 * rank})
    prefill = max(wl.n_new) > 2
    base = di.generate(wl, device=dev)
    # R independently drawn query sets over the same caches: step i uses set i % R, so every
    # step selects and gathers other latent rows (the gathered rows of one step, 75 MB at
    # decode_32k, would otherwise stay in the 129 MB L2 from one step to the next)
    R = max(1, args.query_sets)
    sets = [base] + [di.redraw_queries(base, wl.seed * 1000 + 17 * r) for r in range(1, R)]
    n_q = wl.n_q
    ms, mq = max(wl.seq_lens), max(wl.n_new)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = base["kv8_pool"] if wl.kv_dtype == "fp8" else base["kv_pool"]
    ws = None if prefill else dsa.new_workspace(
        dsa.sfa_workspace_bytes(base["q_sfa"], torch.empty((n_q, wl.K), dtype=torch.int32)), dev)
    li_nb = dsa.li_workspace_bytes(len(wl.seq_lens), wl.K, ms, mq)  # sequences split into units
    li_ws = torch.empty((li_nb,), dtype=torch.uint8, device=dev) if li_nb else None
    bufs, li_args, sfa_args = [], [], []
    for inp in sets:
        o = {"idx": torch.empty((n_q, wl.K), dtype=torch.int32, device=dev),
             "cnt": torch.empty((n_q,), dtype=torch.int32, device=dev),
             "out": torch.empty((n_q, wl.H, wl.d_v), dtype=torch.bfloat16, device=dev),
             "lse": torch.empty((n_q, wl.H), dtype=torch.float32, device=dev)}
        bufs.append(o)
        li_args.append(dsa.li_topk_args(
            inp["q_li"], inp["w"], inp["k_pool"], inp["pt_k"], inp["seq_lens"], inp["q_start"],
            wl.K, q_scale=inp.get("q_scale"), k_scale=inp.get("k_scale"), max_seq_len=ms,
            max_q_per_seq=mq, out_idx=o["idx"], out_cnt=o["cnt"], status=status,
            q_sf=inp.get("q_sf"), k_sf=inp.get("k_sf"), workspace=li_ws))
        sfa_args.append(dsa.sfa_args(
            inp["q_sfa"], kv, inp["pt_kv"], inp["seq_lens"], inp["q_start"], o["idx"],
            softmax_scale=wl.softmax_scale, max_seq_len=ms, max_q_per_seq=mq, out=o["out"],
            lse=o["lse"], status=status, workspace=ws))
    stream = torch.cuda.Stream(device=dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    sfa_entry = lib.dsa_sfa_prefill if prefill else lib.dsa_sfa_decode

    def step(i):
        rc = lib.dsa_li_topk(ctypes.byref(li_args[i % R]), sp)
        rc |= sfa_entry(ctypes.byref(sfa_args[i % R]), sp)
        if rc:
            raise RuntimeError("launch failed: " + dsa.last_error())

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup, R)):
            step(i)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d after warm-up" % int(status.item()))
    cnt_total = sum(int(o["cnt"].sum().item()) for o in bufs) / R
    work = algorithmic(wl, cnt_total)

    # ---- the timed region: exactly K steps, two launches each, no event between the kernels
    # (an event recorded between them would keep the attention kernel from starting its
    # prologue during the indexer's tail: programmatic dependent launch)
    K = args.steps
    e_all = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    # The K steps are captured once as a CUDA graph (the same C-ABI launches, programmatic
    # dependencies included) and replayed once untimed; the timed region replays them once more.
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for i in range(K):
                    step(i)
            graph.replay()
        torch.cuda.synchronize()
    pci = None
    try:
        pr = torch.cuda.get_device_properties(dev)
        pci = "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except Exception:
        pass
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # the clock sampler runs through the timed region and the per-kernel passes after it (a
    # timed region of a few ms would otherwise hold one or two NVML samples)
    clk = ClockSampler(pci)
    with clk:
        with torch.cuda.stream(stream):
            e_all[0].record(stream)
            if graph is not None:
                graph.replay()
            else:
                for i in range(K):
                    step(i)
            e_all[1].record(stream)
        torch.cuda.synchronize()
        clk.mark()
        if world > 1:
            torch.distributed.barrier()
        total_ms = e_all[0].elapsed_time(e_all[1])
        if int(status.item()) != 0:
            raise RuntimeError("device status %d in the timed region" % int(status.item()))
        t = torch.tensor([total_ms], device=dev)
        if world > 1:
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
        value = n_q * world * K / (total_ms / 1000.0)

        # ---- per-kernel durations: each entry point alone, its own event-bracketed pass of
        # args.kernel_reps launches (independent of --steps), median
        NK = max(50, args.kernel_reps)
        li_ms = _median_launch_ms(lib, lib.dsa_li_topk, li_args, sp, stream, NK)
        sfa_ms = _median_launch_ms(lib, sfa_entry, sfa_args, sp, stream, NK)
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the per-kernel passes" % int(status.item()))

    # ---- end to end through host buffers (pinned), copies inside the timed region.
    # Each step's query-side inputs travel host -> device as one packed block and its outputs
    # device -> host as one block, on two copy streams with two device buffer sets, so step n's
    # inputs arrive and step n-1's outputs leave while step n computes.
    e2e = None
    if not args.no_e2e:
        names = [k for k in ["q_li", "q_scale", "q_sf", "w", "q_sfa", "pt_k", "pt_kv", "seq_lens", "q_start"]
                 if base.get(k) is not None]

        def layout(specs):
            offs, off = {}, 0
            for name, shape, dtype in specs:
                nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
                offs[name] = (off, nbytes, shape, dtype)
                off = (off + nbytes + 255) // 256 * 256
            return offs, off

        def carve(block, offs):
            return {k: block[o:o + n].view(dt).view(shape) for k, (o, n, shape, dt) in offs.items()}

        o0 = bufs[0]
        in_offs, in_bytes = layout([(k, tuple(base[k].shape), base[k].dtype) for k in names])
        out_offs, out_bytes = layout([(k, tuple(o0[k].shape), o0[k].dtype) for k in ("idx", "cnt", "out", "lse")])
        host_in = []
        for inp in sets:
            h = torch.zeros(in_bytes, dtype=torch.uint8, pin_memory=True)
            for k, v in carve(h, in_offs).items():
                v.copy_(inp[k].cpu())
            host_in.append(h)
        host_out = [torch.empty(out_bytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
        dev_in = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        dev_out = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        din = [carve(b_, in_offs) for b_ in dev_in]
        dout = [carve(b_, out_offs) for b_ in dev_out]
        li2 = [dsa.li_topk_args(d["q_li"], d["w"], base["k_pool"], d["pt_k"], d["seq_lens"], d["q_start"],
                                wl.K, q_scale=d.get("q_scale"), k_scale=base.get("k_scale"),
                                max_seq_len=ms, max_q_per_seq=mq, out_idx=o["idx"], out_cnt=o["cnt"],
                                status=status, q_sf=d.get("q_sf"), k_sf=base.get("k_sf"),
                                workspace=li_ws)
               for d, o in zip(din, dout)]
        sfa2 = [dsa.sfa_args(d["q_sfa"], kv, d["pt_kv"], d["seq_lens"], d["q_start"], o["idx"],
                             softmax_scale=wl.softmax_scale, max_seq_len=ms, max_q_per_seq=mq,
                             out=o["out"], lse=o["lse"], status=status, workspace=ws)
                for d, o in zip(din, dout)]
        h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        h2d, d2h = in_bytes, out_bytes
        K2 = max(20, K)
        torch.cuda.synchronize()
        for it in range(K2 + 2):
            if it == 2:
                torch.cuda.synchronize()
                if world > 1:
                    torch.distributed.barrier()
                t0 = time.perf_counter()
            s_ = it % 2
            if it >= 2:
                h2d_s.wait_event(ev_done[s_])     # step it-2 no longer reads input set s_
            with torch.cuda.stream(h2d_s):
                dev_in[s_].copy_(host_in[it % R], non_blocking=True)
            ev_in[s_].record(h2d_s)
            stream.wait_event(ev_in[s_])
            if it >= 2:
                stream.wait_event(ev_out[s_])     # step it-2's outputs have left set s_
            rc = lib.dsa_li_topk(ctypes.byref(li2[s_]), sp)
            rc |= sfa_entry(ctypes.byref(sfa2[s_]), sp)
            if rc:
                raise RuntimeError("launch failed: " + dsa.last_error())
            ev_done[s_].record(stream)
            d2h_s.wait_event(ev_done[s_])
            with torch.cuda.stream(d2h_s):
                host_out[s_].copy_(dev_out[s_], non_blocking=True)
            ev_out[s_].record(d2h_s)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        if int(status.item()) != 0:
            raise RuntimeError("device status %d in the end-to-end region" % int(status.item()))
        t = torch.tensor([e2e_s], device=dev)
        if world > 1:
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e = {"value": n_q * world * K2 / float(t.item()), "unit": "tokens/s", "steps": K2,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "copies": "one packed pinned H2D and one D2H per step on two copy streams, double-"
                         "buffered against the compute stream; host input blocks rotate over the "
                         "query sets"}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    hbm, tf, peak_kind = measured_peaks()
    li_gbs = work["k_bytes"] / (li_ms / 1000.0) / 1e9
    sfa_gbs = work["gather_bytes"] / (sfa_ms / 1000.0) / 1e9
    li_tfs = work["li_flop"] / (li_ms / 1000.0) / 1e12
    sfa_tfs = work["sfa_flop"] / (sfa_ms / 1000.0) / 1e12
    step_gbs = work["metric_bytes"] / (total_ms / K / 1000.0) / 1e9
    kernels = {
        "li_topk": {"us": li_ms * 1000.0, "hbm_gbs": li_gbs, "hbm_frac": li_gbs / hbm,
                    "tflops": li_tfs, "tensor_frac": li_tfs / tf,
                    "algorithmic_bytes": work["k_bytes"], "flop": work["li_flop"],
                    "traffic": committed_traffic(args.workload, "li_topk")},
        "sfa": {"us": sfa_ms * 1000.0, "hbm_gbs": sfa_gbs, "hbm_frac": sfa_gbs / hbm,
                "tflops": sfa_tfs, "tensor_frac": sfa_tfs / tf,
                "algorithmic_bytes": work["gather_bytes"], "flop": work["sfa_flop"],
                "traffic": committed_traffic(args.workload, "sfa")},
    }
    # the dominant kernel (longest median launch) against the roofline that bounds it: HBM in
    # decode, the tensor pipe in prefill (4096 tokens share the key pages and most gathered rows)
    dom = "li_topk" if li_ms >= sfa_ms else "sfa"
    kd = kernels[dom]
    if prefill:
        roof = {"kernel": dom, "bound": "tensor", "achieved": kd["tflops"], "peak": tf,
                "unit": "TFLOP/s", "frac": kd["tensor_frac"], "peak_kind": peak_kind + " bf16 burst",
                "traffic": kd["traffic"], "algorithmic_flop": kd["flop"]}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": kd["hbm_gbs"], "peak": hbm,
                "unit": "GB/s", "frac": kd["hbm_frac"], "peak_kind": peak_kind,
                "traffic": kd["traffic"], "algorithmic_bytes": kd["algorithmic_bytes"]}
    roof["timing"] = "median of %d event-bracketed launches of the kernel alone" % NK
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.li_dtype,
        "data": "synthetic",
        "config": {**wl.describe(), "l2": "inputs larger than L2: every step streams %.0f MB of key "
                   "pages, and steps rotate over %d independently drawn query sets, so each step "
                   "gathers other rows of a %.0f MB latent pool" % (
                       work["k_bytes"] / 1e6, R, kv.numel() * kv.element_size() / 1e6),
                   "launch": ("eager C-ABI calls" if graph is None else
                              "one replay of a CUDA graph capturing the K steps' C-ABI calls") +
                             " on one stream, no event between the kernels; the attention kernel "
                             "is a programmatic dependent launch"},
        "roofline": roof,
        "step_hbm": {"metric_bytes": work["metric_bytes"], "achieved_gbs": step_gbs,
                     "frac": step_gbs / hbm, "peak_kind": peak_kind},
        "kernels": kernels,
        "gpu_launches": (4 if li_nb else 2) * K,  # indexer (+ unit plan and merge) + attention
        "clocks": clk.summary(),
    }
    if e2e:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        inp_cpu = di.to_device(base, "cpu")
        rate, cores, sample = oracle_sample_rate(inp_cpu, args.baseline_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_prolog(args):
    """The Indexer Prolog alone (workload prolog_*): per-launch CUDA-event times with an L2 flush
    between launches (the prolog's weights fit in L2; in a model, other layers evict them)."""
    import torch
    import dsa_inputs as di
    import dsa_sparse_attention_li_gb300 as dsa

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = di.preset(args.workload)
    if world > 1:
        wl = di.Workload(**{**wl.__dict__, "seed": wl.seed + 100 * rank})
    inp = di.generate_prolog(wl, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    n_q, F = wl.n_q, wl.H_I * wl.d_I
    mx = wl.li_dtype == "mxfp8"
    q = torch.empty((n_q, wl.H_I, wl.d_I), dtype=torch.float8_e4m3fn if mx else torch.bfloat16, device=dev)
    qsf = torch.empty((n_q, wl.H_I, wl.d_I // 32), dtype=torch.uint8, device=dev) if mx else None
    w = torch.empty((n_q, wl.H_I), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(dsa.prolog_workspace_bytes(inp), 256), dtype=torch.uint8, device=dev)
    lib = dsa.load()
    a = dsa.prolog_args(inp, q_out=q, q_sf=qsf, w_out=w, workspace=ws, status=status)
    stream = torch.cuda.Stream(device=dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 2x the 129 MB L2
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            if lib.dsa_indexer_prolog(ctypes.byref(a), sp):
                raise RuntimeError("prolog launch failed: " + dsa.last_error())
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d after warm-up" % int(status.item()))
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(None) as clk:
        with torch.cuda.stream(stream):
            for i in range(K):
                flush.zero_()
                ev[i][0].record(stream)
                lib.dsa_indexer_prolog(ctypes.byref(a), sp)
                ev[i][1].record(stream)
        torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the timed region" % int(status.item()))
    us = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1000.0
    t = torch.tensor([us], device=dev)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    us = float(t.item())
    if rank != 0:
        return
    # algorithmic bytes: weights once, activations once, quantised q, head weights, key rows
    w_bytes = (F * wl.d_q + wl.d_I * wl.d_model + wl.H_I * wl.d_model) * 2
    a_bytes = n_q * (wl.d_q + wl.d_model) * 2
    o_bytes = n_q * (F * (1 + 1 / 32) if mx else F * 2) + n_q * wl.H_I * 4 + \
        n_q * (wl.d_I * (1 + 1 / 32) if mx else wl.d_I * 2)
    bytes_ = w_bytes + a_bytes + o_bytes
    flop = 2 * n_q * (F * wl.d_q + (wl.d_I + wl.H_I) * wl.d_model)
    hbm, _, peak_kind = measured_peaks()
    gbs = bytes_ / (us * 1e-6) / 1e9
    line = {
        "metric": "indexer_prolog_tokens_per_s", "value": n_q * world / (us * 1e-6), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": us / 1000.0,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.li_dtype,
        "data": "synthetic",
        "config": {"workload": wl.name, "n_q": n_q, "d_q": wl.d_q, "d_model": wl.d_model,
                   "H_I": wl.H_I, "d_I": wl.d_I, "seed": wl.seed,
                   "l2": "L2 flushed (256 MB write) before every timed launch; per-launch CUDA events",
                   "launch": "one C-ABI launch per step (three CTA roles)"},
        "roofline": {"kernel": "prolog", "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "peak_kind": peak_kind, "traffic": committed_traffic(wl.name, "prolog"),
                     "algorithmic_bytes": bytes_},
        "kernels": {"prolog_us": us, "prolog_tflops": flop / (us * 1e-6) / 1e12},
        "gpu_launches": K, "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        cpu = di.to_device(inp, "cpu")
        sub = di.Workload(**{**wl.__dict__, "seq_lens": wl.seq_lens[:2], "n_new": wl.n_new[:2]})
        sample = {k: v for k, v in cpu.items()}
        sample.update(wl=sub, xq=cpu["xq"][:sum(sub.n_new)], x=cpu["x"][:sum(sub.n_new)],
                      seq_lens=cpu["seq_lens"][:2], q_start=cpu["q_start"][:3],
                      pt_k=cpu["pt_k"][:2])
        t0 = time.time()
        oracle.prolog(sample)
        dt = time.time() - t0
        line["cpu_baseline"] = {"value": sub.n_q / dt, "unit": "tokens/s",
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": "%d tokens of the workload" % sub.n_q}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.workload.startswith("prolog"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the oracle arm times the decode path; the prolog has its own "
                              "cpu_baseline"}))
            return
        run_prolog(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
