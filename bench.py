"""Benchmark of mha_prefill on GB300: unmasked TFLOP/s and tokens/s, % of the
dense-BF16 tensor peak, roofline of the attention kernel, an end-to-end
number through the C ABI with host buffers, and the CPU oracle as a baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...    # the CPU oracle as the reference arm
  python bench.py ... --log runs.jsonl [--resume] [--sample-rows N]

--log appends the printed line to a file as well; with --resume a run whose
(workload, seed, implementation, GPU count) the file already holds is not
repeated: its logged line is printed again, so a sweep over workloads that
was killed part way can be restarted with the same commands.

One step = one tsk_mha_prefill call (scheduler pre-pass + attention kernel)
over the whole workload, inputs resident in HBM.  L2 is flushed before every
timed step: a 256 MB write, then a 256 MB read of another buffer, so that
the written lines are evicted (written back to HBM) before the step starts
and the step finds a cold L2 without paying for the flush's write-backs;
only the step itself is inside the CUDA events.  Under torchrun (N > 1) every rank runs an independent replica on its
own GPU (the operation has no cross-GPU exchange); value = all ranks' FLOPs /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
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

import inputgen  # noqa: E402

DEFAULT_WORKLOAD = "causal_4x4096_h64kv8"
METRIC = "mha_prefill unmasked TFLOP/s and tokens/s on 1 GB300; % of dense-BF16 peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
NVSMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            def find(keys):
                for k in keys:
                    if k in d and isinstance(d[k], (int, float)):
                        return float(d[k])
                for v in d.values():
                    if isinstance(v, dict):
                        for k in keys:
                            if k in v and isinstance(v[k], (int, float)):
                                return float(v[k])
                return None
            bf = find(["bf16_tflops"])
            if bf:
                return {"bf16_tflops": bf,
                        "bf16_tflops_sustained": find(["bf16_tflops_sustained"]) or bf,
                        "hbm_gbs": find(["hbm_gbs"]) or FALLBACK_PEAKS["hbm_gbs"]}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(D=64, decode=False, fp8=False):
    """Hash of the device sources the timed kernel is built from (the host file
    and the other kernels' own headers excluded)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gqa_attention_prefill_gb300", "csrc")
    files = ["ptx.cuh", "schedule.cuh", "attention.cuh"]
    files += (["decode.cuh"] if decode else
              ["attention_fp8.cuh"] + (["attention_d128.cuh"] if D == 128 else []) if fp8 else
              ["attention_d128.cuh"] if D == 128 else [])
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, D=64, decode=False, fp8=False):
    """Per-launch DRAM bytes of the timed kernel from a committed ncu summary,
    if it was taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(workload)
        if e and e.get("kernel_source_hash") == kernel_source_hash(D, decode, fp8):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix=f"tsk_clocks_gpu{self.gpu}_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={NVSMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_rate(w, seconds_target, seed_stream=77, keep=None, rows=0):
    """Times the CPU oracle on a uniform sample of (token, head) rows of `w`
    sized for about `seconds_target` of CPU work (or of `rows` rows, if
    given).  Returns (flop/s, rows, seconds, threads, flops)."""
    import oracle
    G = w.Hq // w.Hkv
    T = w.total_tokens
    cu = w.cu_seqlens

    def rows_flops(n):
        r = inputgen.uniform_int(w.seed, seed_stream + n, n, 0, T * w.Hq - 1)
        t = (r // w.Hq).astype(np.int64)
        h = (r % w.Hq).astype(np.int32)
        s = np.searchsorted(cu, t, side="right") - 1
        pos = t - cu[s]
        if w.cu_seqlens_k is not None:   # key position of the query (cache prefix first)
            pos = pos + (np.diff(w.cu_seqlens_k)[s] - np.diff(cu)[s])
        nk = pos + 1 if w.window <= 0 else np.minimum(pos + 1, w.window)
        return t, h, float(4.0 * w.D * nk.sum())

    if rows > 0:
        n2 = int(rows)
    else:
        n = 2048
        t, h, fl = rows_flops(n)
        t0 = time.perf_counter()
        oracle.run_workload(w, rows=(t, h))
        dt = time.perf_counter() - t0
        n2 = int(min(4_000_000, max(n, n * seconds_target / max(dt, 1e-3))))
    t, h, fl = rows_flops(n2)
    t0 = time.perf_counter()
    ro, rl, thr = oracle.run_workload(w, rows=(t, h))
    dt = time.perf_counter() - t0
    if keep is not None:   # the sampled rows and the oracle's values for them
        keep.update(t=t, h=h, out=ro, lse=rl)
    return fl / dt, n2, dt, thr, fl


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def roofline_of(flops, alg_bytes, kernel_s, peaks, peak_src, fp8=False):
    """The tensor-core and HBM roofs of one launch (algorithmic FLOP and bytes
    over the kernel time), and the binding one: HBM when the arithmetic
    intensity is below the ridge point (peak FLOP/s over peak bytes/s), the
    tensor cores above it."""
    # E4M3 inputs: QK^T (half the FLOP) runs as an E4M3 contraction at twice the
    # dense bf16 rate (the nominal fp8/bf16 ratio), PV in bf16 at the bf16 rate,
    # so the roof for the whole is 1 / (1/4 + 1/2) = 4/3 of the bf16 peak.
    tensor_peak = peaks["bf16_tflops"] * (4.0 / 3.0 if fp8 else 1.0)
    roofs = {
        "tensor": {"achieved": flops / kernel_s / 1e12, "peak": tensor_peak, "unit": "TFLOP/s",
                   "frac": flops / kernel_s / 1e12 / tensor_peak,
                   # (the same against the peak measured over a seconds-long loop
                   # under the power cap)
                   "frac_of_sustained": flops / kernel_s / 1e12 /
                                        (peaks["bf16_tflops_sustained"] * (4.0 / 3.0 if fp8 else 1.0)),
                   "peak_source": (f"{peak_src} dense bf16 (burst) x 4/3 (E4M3 QK^T at 2x, "
                                   "bf16 PV)" if fp8 else f"{peak_src} dense bf16 (burst)")},
        "hbm": {"achieved": alg_bytes / kernel_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": alg_bytes / kernel_s / 1e9 / peaks["hbm_gbs"],
                "peak_source": f"{peak_src} HBM copy bandwidth"},
    }
    intensity = flops / alg_bytes
    ridge = tensor_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    bound = "hbm" if intensity < ridge else "tensor"
    r = roofs[bound]
    roofline = {"bound": bound, "achieved": r["achieved"], "peak": r["peak"], "unit": r["unit"],
                "frac": r["frac"], "traffic": None, "peak_source": r["peak_source"],
                "algorithmic_bytes": alg_bytes, "algorithmic_flop": flops,
                "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge}
    return roofline, roofs


def config_dict(w, ws):
    """The workload description both arms print (identical for the same run)."""
    kv = w.cu_seqlens_k is not None
    return {"workload": w.name, "seed": w.seed,
            "seqlens": w.seqlens if len(w.seqlens) <= 8 else f"{len(w.seqlens)} seqs",
            "total_tokens": w.total_tokens,
            "key_lengths": (w.seqlens_k if kv and len(w.seqlens_k) <= 8 else
                            (f"{len(w.seqlens_k)} seqs, {w.total_keys} keys" if kv else None)),
            "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "window": w.window, "scale": w.scale,
            "sinks": w.sinks is not None, "lse": True,
            "inputs": "fp8 e4m3 (per-tensor scales)" if w.fp8 is not None else "bf16",
            "l2": "flushed before every timed GPU step (256 MB write, then 256 MB read)",
            "parallelism": "replicas" if ws > 1 else "single GPU"}


def run_key(workload, seed, impl, n_gpus):
    """What identifies a run in a --log file."""
    return f"{workload}|{seed}|{impl}|{n_gpus}"


def line_key(line):
    c = line.get("config") or {}
    return run_key(c.get("workload"), c.get("seed"), line.get("impl", "ours"), line.get("n_gpus"))


def logged_line(path, key):
    """The last line of the log `path` with this run key, or None.  Lines that
    do not parse (one cut short by a killed run) are skipped."""
    if not path or not os.path.exists(path):
        return None
    found = None
    with open(path) as f:
        for text in f:
            text = text.strip()
            if not text:
                continue
            try:
                d = json.loads(text)
            except ValueError:
                continue
            if isinstance(d, dict) and line_key(d) == key:
                found = text
    return found


def emit(line, log=None):
    """Print the result line (and append it to the log file, if any)."""
    text = json.dumps(line)
    print(text, flush=True)
    if log:
        with open(log, "a") as f:
            f.write(text + "\n")


def parity_stats(gpu_out, gpu_lse, ref_out, ref_lse):
    """max/mean |d| of sampled output rows ([n, D]) and max |d| of their LSE ([n])."""
    o = gpu_out.astype(np.float64)
    d = np.abs(o - ref_out)
    dl = np.abs(gpu_lse.astype(np.float64) - ref_lse)
    return {"rows": int(len(o)), "out_max_abs": float(d.max()), "out_mean_abs": float(d.mean()),
            "lse_max_abs": float(dl.max()), "finite": bool(np.isfinite(o).all())}


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    w = inputgen.config(args.workload, seed=args.seed)
    flops_total = w.unmasked_flops()
    # each step: the oracle on a bounded row sample (~3 s of CPU work)
    for _ in range(args.warmup):
        oracle_rate(w, 0.5)
    rates, step_s, rows, thr = [], [], 0, 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        r, n, dt, thr, fl = oracle_rate(w, 3.0)
        step_s.append(time.perf_counter() - t0)
        rates.append(r)
        rows = n
    value = statistics.median(rates) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        # (the launch's GPU count, as in the GPU arm's line; the oracle itself
        # runs on the host's cores, see cpu_baseline)
        "n_gpus": ws, "runs_on": "host CPU cores", "steps": args.steps, "warmup": args.warmup,
        # measured wall time of one step (a bounded row sample, rate calibration included)
        "ms_per_step": statistics.mean(step_s) * 1e3,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": config_dict(w, ws),
        "step": f"the CPU oracle on {rows} uniform (token, head) rows of the workload",
        "ms_per_full_workload_extrapolated": flops_total / (value * 1e12) * 1e3,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"{rows} uniform (token, head) rows per step of {w.name}, "
                                   f"~{statistics.mean(step_s):.1f} s each"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    emit(line, args.log)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(inputgen.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sample-rows", type=int, default=0,
                    help="rows of the oracle sample that checks the output (default: sized "
                         "by --cpu-seconds)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--log", default=None, help="also append the JSON line to this file")
    ap.add_argument("--resume", action="store_true",
                    help="with --log: print the logged line of this run instead of repeating it")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    ws, rank, local = dist_env()
    if args.resume and args.log:
        done = logged_line(args.log, run_key(args.workload, args.seed, args.impl, ws))
        if done is not None:
            if rank == 0:
                print(done, flush=True)
            return 0
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo", init_method="env://")
    if args.impl == "reference":
        rc = run_reference(args, ws, rank)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return rc

    import torch
    import gqa_attention_prefill_gb300 as pkg
    from gqa_attention_prefill_gb300 import build as cuda_build
    if not os.path.exists(pkg.library_path()):
        cuda_build.build()
    lib = pkg.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    w = inputgen.config(args.workload, seed=args.seed + rank)
    T, Hq, Hkv, D = w.total_tokens, w.Hq, w.Hkv, w.D
    flops = w.unmasked_flops()

    # host (pinned) and device copies
    fp8 = w.fp8 is not None  # E4M3 inputs with per-tensor scales
    if fp8:
        h_q, h_k, h_v = (torch.from_numpy(w.fp8[n]).pin_memory() for n in ("q", "k", "v"))
    else:
        h_q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).pin_memory()
        h_k = torch.from_numpy(w.k.view(np.int16)).view(torch.bfloat16).pin_memory()
        h_v = torch.from_numpy(w.v.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_s = torch.from_numpy(w.sinks).pin_memory()
    h_cu = torch.from_numpy(w.cu_seqlens).pin_memory()
    kvcache = w.cu_seqlens_k is not None
    decode = kvcache and all(L == 1 for L in w.seqlens)  # one query token per sequence
    h_cuk = torch.from_numpy(w.cu_seqlens_k if kvcache else w.cu_seqlens).pin_memory()
    q, k, v = h_q.to(dev), h_k.to(dev), h_v.to(dev)
    sinks, cu, cuk = h_s.to(dev), h_cu.to(dev), h_cuk.to(dev)
    out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)  # bf16 for every input type
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    evict = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()   # 256 MB of dirty lines replace the L2's contents
        evict.sum()     # a 256 MB read writes them back before the next step

    def step(o=out, l=lse, qq=q, kk=k, vv=v, ss=sinks, cc=cu, ck=cuk):
        if fp8:
            f = w.fp8
            rc = pkg.tsk_mha_prefill_fp8(qq, kk, vv, f["q_scale"], f["k_scale"], f["v_scale"], ss,
                                         cc, w.num_seqs, T, Hq, Hkv, D, w.window, w.scale, o, l,
                                         stream)
        elif decode:
            rc = pkg.tsk_mha_decode_kvcache(qq, kk, vv, ss, ck, w.num_seqs, w.total_keys,
                                            max(w.seqlens_k), Hq, Hkv, D, w.window, w.scale, o, l,
                                            stream)
        elif kvcache:
            rc = pkg.tsk_mha_prefill_kvcache(qq, kk, vv, ss, cc, ck, w.num_seqs, T, w.total_keys,
                                             Hq, Hkv, D, w.window, w.scale, o, l, stream)
        else:
            rc = pkg.tsk_mha_prefill(qq, kk, vv, ss, cc, w.num_seqs, T, Hq, Hkv, D, w.window,
                                     w.scale, o, l, stream)
        if rc != 0:
            raise pkg.TskError(rc, "tsk_mha_prefill")

    pkg.tsk_profile_enable(True)
    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    st = pkg.tsk_get_device_status(stream)
    if st != 0:
        raise pkg.TskError(st, "device status after warm-up")

    # ---------------------------------------------------------------- timed
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    attn_ms, pre_ms = [], []
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                      else local) as clk:
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
            a, b = pkg.tsk_profile_read()   # waits for this step's events
            pre_ms.append(a)
            attn_ms.append(b)
        torch.cuda.synchronize()
    barrier(ws)
    step_ms = [s.elapsed_time(e) for s, e in ev]
    st = pkg.tsk_get_device_status(stream)
    if st != 0:
        raise pkg.TskError(st, "device status after timed steps")
    ms = reduce_max(sum(step_ms) / len(step_ms), ws)
    attn_avg = reduce_max(sum(attn_ms) / len(attn_ms), ws)
    value = flops * ws / (ms * 1e-3) / 1e12

    # ---------------------------------------------------------------- end to end
    h_out = torch.empty((T, Hq, D), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty((T, Hq), dtype=torch.float32).pin_memory()
    d_q, d_k, d_v = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    d_s, d_cu, d_cuk = torch.empty_like(sinks), torch.empty_like(cu), torch.empty_like(cuk)
    pkg.tsk_profile_enable(False)

    # Plain prefill goes through the host-buffer entry point (the library
    # overlaps chunked copies with the attention); the other paths copy with
    # torch and call the device entry point.
    host_api = not (fp8 or kvcache)

    def e2e_step():
        if host_api:
            rc = pkg.tsk_mha_prefill_host(h_q, h_k, h_v, h_s, h_cu, w.num_seqs, T, Hq, Hkv, D,
                                          w.window, w.scale, h_out, h_lse, stream)
            if rc != 0:
                raise pkg.TskError(rc, "tsk_mha_prefill_host")
            return
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        d_s.copy_(h_s, non_blocking=True)
        d_cu.copy_(h_cu, non_blocking=True)
        if kvcache:
            d_cuk.copy_(h_cuk, non_blocking=True)
        step(out, lse, d_q, d_k, d_v, d_s, d_cu, d_cuk if kvcache else d_cu)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for _ in range(args.e2e_steps):
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e_ms.append(e0.elapsed_time(e1))
    e2e_ms = reduce_max(sum(e_ms) / len(e_ms), ws)
    h2d = sum(x.numel() * x.element_size() for x in (h_q, h_k, h_v, h_s, h_cu)) + \
        (h_cuk.numel() * 4 if kvcache else 0)
    d2h = h_out.numel() * 2 + h_lse.numel() * 4
    # the e2e outputs must equal the resident-input outputs
    torch.cuda.synchronize()
    same = torch.equal(h_out.view(torch.int16), out.cpu().view(torch.int16))

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    kernel_s = attn_avg * 1e-3
    alg_bytes = w.algorithmic_bytes()
    kernel_name = ("decode_split_kernel<%d> (merging its splits)" % D if decode else
                   "attention_fwd_d128_kernel<0, true> (E4M3 Q/K)" if fp8 and D == 128 else
                   "attention_fwd_fp8_kernel" if fp8 else
                   "attention_fwd_d128_kernel" if D == 128 else
                   "attention_fwd_kernel<true>" if 0 < w.window <= 512 else
                   "attention_fwd_kernel<false>")
    traffic = ncu_traffic(w.name, D, decode, fp8)
    roofline, roofs = roofline_of(flops, alg_bytes, kernel_s, peaks, peak_src, fp8)
    roofline.update(traffic=traffic, kernel=kernel_name)
    # Exponentials: one per allowed (query, key, head) triple, i.e. the
    # unmasked FLOP over 4 D, against the measured rate of the exponential
    # instruction the softmax uses.
    ex2_peak = pkg.tsk_bench_ex2_rate(stream)
    exps = flops / (4.0 * D)
    exp_roof = {"achieved": exps / kernel_s / 1e9, "peak": ex2_peak / 1e9, "unit": "Gexp/s",
                "frac": exps / kernel_s / ex2_peak,
                "peak_source": "measured ex2.approx.f32 throughput (tsk_bench_ex2_rate, this run)",
                "note": "algorithmic exponentials (unmasked scores); the kernel also evaluates "
                        "masked positions of tiles that straddle the diagonal or window edge"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 QK^T, bf16 PV (fp32 accumulation)" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, fp32 sinks)",
        "config": config_dict(w, ws),
        "tokens_per_s": T * ws / (ms * 1e-3),
        "pct_of_bf16_peak": value / peaks["bf16_tflops"] * 100.0,
        "pct_of_bf16_sustained_peak": value / peaks["bf16_tflops_sustained"] * 100.0,
        "unmasked_flop_per_step": flops,
        "attention_kernel_ms": attn_avg, "prepass_kernel_ms": sum(pre_ms) / len(pre_ms),
        "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
        "roofline": roofline,
        "roofs": roofs,
        "exp": exp_roof,
        "e2e": {"value": flops * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "matches_resident_run": bool(same),
                "via": ("tsk_mha_prefill_host (pinned host buffers; chunked copies overlapped "
                        "with the attention)" if host_api else
                        "pinned host buffers copied by torch, then the device entry point")},
        # decode: offset check + split kernel; FP8: scheduler + V transpose +
        # attention; otherwise tsk_mha_prefill's scheduler + attention
        "gpu_launches": args.steps * (2 if decode else 3 if fp8 else pkg.tsk_kernels_per_call()),
        "clocks": clk.summary(),
        "kernel_source_hash": kernel_source_hash(D, decode, fp8),
    }
    if not args.no_cpu_baseline:
        # The CPU oracle on a bounded uniform sample of (token, head) rows: its
        # rate is the baseline, and its values for those rows check the output
        # of the last timed step.
        keep = {}
        r, n, dt, thr, fl = oracle_rate(w, args.cpu_seconds, keep=keep, rows=args.sample_rows)
        line["cpu_baseline"] = {"value": r / 1e12, "unit": "TFLOP/s", "cores": thr,
                                "kind": "oracle",
                                "sample": f"{n} uniform (token, head) rows of {w.name} "
                                          f"({fl / 1e9:.1f} GFLOP, {dt:.1f} s)"}
        ti = torch.from_numpy(keep["t"]).to(dev)
        hi = torch.from_numpy(keep["h"].astype(np.int64)).to(dev)
        g_out = out[ti, hi].float().cpu().numpy()
        g_lse = lse[ti, hi].cpu().numpy()
        line["parity"] = dict(
            parity_stats(g_out, g_lse, keep["out"], keep["lse"]),
            of="the timed run's output (last step) at the cpu_baseline's sampled rows, "
               "against the CPU oracle",
            tolerance={"out_max_abs": 2e-2, "out_mean_abs": 2e-3, "lse_max_abs": 1e-3})
    emit(line, args.log)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
