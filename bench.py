#!/usr/bin/env python3
"""Benchmark: Sparse-Flash-MLA Softmax-L1Norm forward on GB300.

One step = one launch of the fused kernel over the whole workload (gather,
Q.K^T on the tensor cores, scale/mask/exp against the LSE, head-group mean,
store).  Default workload: the DeepSeek-V3.2-like sparse causal
configuration (BSND, B=1, S1=S2=4096, N1=128, D=512, bf16, top-2048 of the
causally visible keys, right-down causal mask).

Prints ONE JSON line (rank 0).  ``value`` is selected query-key pairs per
second (a pair = one 512-long per-head dot product on a kept slot), whole job.

  python bench.py [--steps K] [--warmup W] [--config N] [--impl ours|reference]
  torchrun --nproc-per-node N bench.py --gpus N ...   (independent replicas)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "selected q.k pairs/s (Softmax-L1Norm forward, whole job)"
UNIT = "pairs/s"
L2_FLUSH_BYTES = 512 << 20   # > the 129 MB L2
# Per L1-norm kernel: its ncu DRAM-traffic summary and the sources it is
# built from (its own file and the device code the two kernels share).
_CSRC = os.path.join(ROOT, "softmax_l1_norm_gb300", "csrc")
KERNELS = {
    "smla_fused_kernel": (os.path.join(ROOT, "profiles", "smla_fused_kernel_dsv32_traffic.txt"),
                          [os.path.join(_CSRC, f) for f in ("smla_kernel.cu", "smla_device.cuh")]),
    "smla_pair_kernel": (os.path.join(ROOT, "profiles", "smla_pair_kernel_dsv32_traffic.txt"),
                         [os.path.join(_CSRC, f) for f in ("smla_pair.cu", "smla_device.cuh")]),
}


# ----------------------------------------------------------------------------
def workload_numbers(w):
    """Pairs, FLOPs and bytes of one pass over the workload.

    ``bytes_`` counts every gathered key row as read (the roofline the work
    was specified against); ``compulsory`` counts each tensor once -- the
    keys any slot refers to, q, the LSE, the indices and the output -- which
    is what a pass must move between HBM and the chip at the least."""
    valid = w.valid_slot_count()
    pairs = valid * w.G
    flops = 2 * w.head_dim * pairs
    n = w.n_tokens
    bytes_ = {
        "k_gathered": valid * w.head_dim * 2,
        "q": n * w.G * w.head_dim * 2,
        "lse": n * w.G * 4,
        "out": n * w.out_width * 4,
        "indices": 0 if w.sparse_indices is None else n * w.topk * 4,
        "topk_length": 0 if w.topk_length is None else n * 4,
    }
    compulsory = dict(bytes_)
    compulsory.pop("k_gathered")
    compulsory["k_unique"] = unique_key_rows(w) * w.head_dim * 2
    return pairs, flops, bytes_, compulsory


def unique_key_rows(w):
    """Key rows that at least one kept slot refers to."""
    tab = w.token_table()
    n_rows = int(w.k_bits.reshape(-1, w.head_dim).shape[0])
    if n_rows == 0:
        return 0
    seen = np.zeros(n_rows, dtype=bool)
    if w.sparse_indices is None:
        vis = W.visible_count(tab[:, 1], tab[:, 2], tab[:, 4], w.mask_mode)
        vis = np.minimum(vis, w.out_width)
        for b, q0, Sq, k0, Sk in w.sequences():
            if Sq > 0:
                seen[k0:k0 + int(vis[q0:q0 + Sq].max())] = True
        return int(seen.sum())
    idx = w.sparse_indices.reshape(w.n_tokens, w.topk).astype(np.int64)
    Sk = tab[:, 4:5]
    ok = (idx >= 0) & (idx < Sk)
    if w.mask_mode == 3:
        ok &= idx <= (tab[:, 1:2] + Sk - tab[:, 2:3])
    if w.topk_length is not None:
        ok &= np.arange(w.topk)[None, :] < w.topk_length.reshape(w.n_tokens, 1).astype(np.int64)
    seen[(tab[:, 3:4] + idx)[ok]] = True
    return int(seen.sum())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def l1_kernel_name(plan):
    """The kernel a plan's L1-norm launch runs."""
    return "smla_pair_kernel" if plan.info.cta_pairs > 0 else "smla_fused_kernel"


def kernel_sha(kernel="smla_fused_kernel"):
    """Hash of a kernel's sources with comments and blank lines removed, so
    that edits to comments keep the profiled traffic valid."""
    import re
    src = ""
    for path in KERNELS[kernel][1]:
        with open(path, encoding="utf-8") as f:
            src += f.read() + "\n"
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    code = "\n".join(line.rstrip() for line in src.splitlines() if line.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def profiled_traffic(config_name, kernel="smla_fused_kernel"):
    """DRAM bytes per launch of `kernel` from its committed ncu summary, if
    that was taken on the current source of the kernel and on this
    workload; else None."""
    path = KERNELS[kernel][0]
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_sha256_16") != kernel_sha(kernel) or kv.get("workload") != config_name:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="smla_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, smax, reasons, n = [], [], set(), 0
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
                n += 1
                for name, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": float(np.median(load)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": n}


# ----------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def all_max(x, world, device=None):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------
_ORACLE_CHILD = r"""
import json, sys, time
import numpy as np
P = json.loads(sys.argv[1])
sys.path.insert(0, P["root"])
import workloads as W, oracle
w = W.make_config(P["config"], seq_len=P.get("seq_len"))
kw = dict(dtype=w.dtype, sparse_indices=w.sparse_indices, topk_length=w.topk_length,
          cu_seqlens_q=w.cu_seqlens_q, cu_seqlens_k=w.cu_seqlens_k, softmax_scale=w.softmax_scale,
          max_seqlen_k=w.max_seqlen_k, mask_mode=w.mask_mode, layout=w.layout)
tab = w.token_table()
def kept(t):
    b, r, Sq, k0, Sk = (int(x) for x in tab[t])
    if w.sparse_indices is None:
        return min(Sk, max(0, r + Sk - Sq + 1)) if w.mask_mode == 3 else Sk
    idx = w.sparse_indices.reshape(w.n_tokens, -1)[t].astype(np.int64)
    ok = (idx >= 0) & (idx < Sk)
    if w.mask_mode == 3:
        ok &= idx <= r + Sk - Sq
    if w.topk_length is not None:
        ok &= np.arange(len(idx)) < int(w.topk_length.reshape(-1)[t])
    return int(ok.sum())
rows = np.random.Generator(np.random.PCG64(P["seed"])).permutation(w.n_tokens).tolist()
pos = 0
def one(n):
    global pos
    pairs = 0
    t0 = time.perf_counter()
    for _ in range(n):
        t = rows[pos % len(rows)]
        pos += 1
        oracle.softmax_l1_norm_rows(w.q_bits, w.k_bits, w.softmax_lse, [t], **kw)
        pairs += kept(t) * w.G
    return pairs, time.perf_counter() - t0
res = {"warmup": [], "steps": []}
per_row = None
for _ in range(P["warmup"]):
    p, dt = one(1)
    per_row = dt if per_row is None else min(per_row, dt)
    res["warmup"].append([1, p, dt])
n = max(1, int(P["step_seconds"] / max(per_row or P["step_seconds"], 1e-6)))
for _ in range(P["steps"]):
    p, dt = one(n)
    res["steps"].append([n, p, dt])
print(json.dumps(res))
"""


def cpu_oracle_run(config, warmup, steps, step_seconds, threads, seed=0, seq_len=None):
    """Time the CPU oracle, as it stands, on bounded samples of the workload's
    rows: ``warmup`` single rows, then ``steps`` steps of about
    ``step_seconds`` each.  Runs in a child process so the BLAS thread count
    is fixed before numpy loads and no CUDA context is involved."""
    params = json.dumps({"root": ROOT, "config": config, "seed": seed, "warmup": max(1, warmup),
                         "steps": steps, "step_seconds": step_seconds, "seq_len": seq_len})
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, "-c", _ORACLE_CHILD, params], capture_output=True, text=True,
                       env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"cpu oracle run failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: the
    implementer and part numbers), or None."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return None
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"Arm implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return None


# ----------------------------------------------------------------------------
def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step runs it on a bounded
    sample of the same workload (rank 0 only; other ranks exit at once)."""
    if rank != 0:
        return 0
    threads = host_threads()
    # every step is a bounded sample; the whole run stays within --ref-total-seconds
    step_s = max(0.02, min(args.ref_step_seconds, args.ref_total_seconds / max(1, args.steps)))
    r = cpu_oracle_run(args.config, args.warmup, args.steps, step_s, threads, seq_len=args.seq_len)
    rows = sum(s[0] for s in r["steps"])
    pairs = sum(s[1] for s in r["steps"])
    secs = sum(s[2] for s in r["steps"])
    name = W.CONFIG_NAMES[args.config] if args.seq_len is None else \
        W.make_config(args.config, seq_len=args.seq_len).name
    value = pairs / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": name, "note": "CPU fp64 oracle on a bounded random sample of rows per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"{rows} random rows of {name} over {args.steps} steps "
                                   f"(~{step_s:.2f}s each)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class L2Flush:
    """Between timed launches: write 512 MB (evicts all of the 129 MB L2),
    then read a separate 256 MB buffer, so that the lines the write left
    dirty are written back to HBM here and not charged to the next timed
    launch.  The timed kernel starts with none of its data in L2."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.float32, device=device)
        self.acc = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.acc)


def step_stats(times_ms):
    t = np.asarray(times_ms, dtype=np.float64)
    return {"median": float(np.median(t)), "mean": float(t.mean()), "min": float(t.min()),
            "max": float(t.max()), "p10": float(np.percentile(t, 10)), "p90": float(np.percentile(t, 90)),
            "n": int(t.size)}


def timed_launches(fn, steps, stream, flush):
    """``steps`` launches of ``fn``, each after an L2 flush, each bracketed by
    CUDA events on ``stream``; returns the per-launch times in ms."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def roofline_block(flops, compulsory_bytes, seconds, hbm_gbs, bf16_tf, src, traffic=None):
    """The binding bound: the larger of the tensor time and the time to move
    the compulsory bytes at the measured HBM bandwidth."""
    t_tc = flops / (bf16_tf * 1e12)
    t_hbm = compulsory_bytes / (hbm_gbs * 1e9)
    if t_tc >= t_hbm:
        bound, achieved, peak, unit = "tensor", flops / seconds / 1e12, bf16_tf, "TFLOP/s"
    else:
        bound, achieved, peak, unit = "hbm", compulsory_bytes / seconds / 1e9, hbm_gbs, "GB/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": traffic, "peak_source": f"{src} (MEASURED_PEAKS.json: bf16 burst, HBM copy)",
            "roofline_ms": 1000 * max(t_tc, t_hbm), "kernel_ms": 1000 * seconds,
            "tensor_ms": 1000 * t_tc, "compulsory_hbm_ms": 1000 * t_hbm,
            "compulsory_bytes": int(compulsory_bytes)}


def gathered_bytes_block(alg_bytes, seconds, hbm_gbs, t_tc_s):
    """A second roofline: every gathered key row counted as HBM traffic (with
    q, lse, indices and the output).  The keys of these workloads fit in L2,
    so this bound does not bind; kept for reference only."""
    t_hbm = alg_bytes / (hbm_gbs * 1e9)
    return {"bytes_counted": int(alg_bytes), "hbm_ms": 1000 * t_hbm, "tensor_ms": 1000 * t_tc_s,
            "roofline_ms": 1000 * max(t_hbm, t_tc_s), "kernel_ms": 1000 * seconds,
            "frac_of_this_bound": 1000 * max(t_hbm, t_tc_s) / (1000 * seconds),
            "note": "counts every gathered key row as DRAM traffic; the keys are L2-resident, "
                    "so a fraction above 1 here does not mean skipped work"}


def device_inputs(w, device):
    import torch
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    host = {
        "q": torch.from_numpy(w.q_bits.view(np.int16)).view(tdt),
        "k": torch.from_numpy(w.k_bits.view(np.int16)).view(tdt),
        "lse": torch.from_numpy(np.ascontiguousarray(w.softmax_lse, dtype=np.float32)),
        "indices": None if w.sparse_indices is None else torch.from_numpy(w.sparse_indices),
        "topk_length": None if w.topk_length is None else torch.from_numpy(w.topk_length),
    }
    dev = {k: (None if v is None else v.to(device)) for k, v in host.items()}
    return host, dev


def make_plan(smla, w):
    return smla.Plan(layout=w.layout, dtype=w.dtype, num_heads_q=w.G, batch_size=w.batch,
                     max_seqlen_q=w.max_seqlen_q if w.layout == "BSND" else 0,
                     max_seqlen_k=w.k_bits.shape[1] if w.layout == "BSND" else w.max_seqlen_k,
                     topk=w.topk, mask_mode=w.mask_mode, softmax_scale=w.softmax_scale,
                     has_topk_length=w.topk_length is not None,
                     cu_seqlens_q=None if w.cu_seqlens_q is None else w.cu_seqlens_q.tolist(),
                     cu_seqlens_k=None if w.cu_seqlens_k is None else w.cu_seqlens_k.tolist())


def other_config_line(smla, n, steps, device, stream, flush, gpu_id=None):
    """One configuration other than the headline, timed the same way (after
    the headline's timed region): median ms per launch and the roofline."""
    import torch
    w = W.make_config(n)
    pairs, flops, bytes_, compulsory = workload_numbers(w)
    _, dev = device_inputs(w, device)
    plan = make_plan(smla, w)
    out = torch.empty(plan.output_shape, dtype=torch.float32, device=device)

    def fn():
        plan.run(dev["q"], dev["k"], dev["lse"], sparse_indices=dev["indices"],
                 topk_length=dev["topk_length"], out=out, stream=stream)

    for _ in range(3):
        flush()
        fn()
    torch.cuda.synchronize(device)
    with ClockSampler(gpu_id if gpu_id is not None else device.index) as clocks:
        time.sleep(0.3)  # the sampler's first readings
        times = timed_launches(fn, steps, stream, flush)
    code, flags = plan.status(stream)
    if code != smla.SMLA_OK:
        raise RuntimeError(f"config {n}: device status {code} flags {flags}")
    st = step_stats(times)
    hbm_gbs, bf16_tf, src = load_peaks()
    sec = st["median"] / 1000.0
    line = {"workload": w.name, "ms_per_launch": st, "pairs_per_s": pairs / sec, "tflops": flops / sec / 1e12,
            "pairs": pairs, "flops": flops,
            "roofline": dict(roofline_block(flops, sum(compulsory.values()), sec, hbm_gbs, bf16_tf, src),
                             kernel=l1_kernel_name(plan)),
            "clocks": clocks.summary(),
            "gathered_bytes_roofline": gathered_bytes_block(sum(bytes_.values()), sec, hbm_gbs,
                                                            flops / (bf16_tf * 1e12)),
            "plan": {k: v for k, v in plan.info.as_dict().items() if k in ("num_ctas", "num_items", "stages",
                                                                            "mma_n", "rows_per_item", "mma_issuers",
                                                                            "cta_pairs", "split_tiles",
                                                                            "split_items")}}
    del plan, dev, out
    torch.cuda.empty_cache()
    return line


def run_ours(args, world, rank, local):
    import torch

    import softmax_l1_norm_gb300 as smla

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)

    w = W.make_config(args.config, seq_len=args.seq_len)
    name = w.name
    pairs, flops, bytes_, compulsory = workload_numbers(w)
    alg_bytes = sum(bytes_.values())
    comp_bytes = sum(compulsory.values())

    host, dev = device_inputs(w, device)
    plan = make_plan(smla, w)
    out = torch.empty(plan.output_shape, dtype=torch.float32, device=device)
    flush = L2Flush(device)

    def step():
        plan.run(dev["q"], dev["k"], dev["lse"], sparse_indices=dev["indices"],
                 topk_length=dev["topk_length"], out=out, stream=stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(device)
    code, flags = plan.status(stream)
    if code != smla.SMLA_OK:
        raise RuntimeError(f"device status {code} flags {flags} during warm-up")
    if not bool(torch.isfinite(out).all()):
        raise RuntimeError("non-finite output")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(device).uuid)
        if not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        pass
    barrier(world, device)
    torch.cuda.synchronize(device)
    with ClockSampler(gpu_uuid if gpu_uuid else local) as clocks:
        time.sleep(0.3)
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush()                # outside the events
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
        wall = time.perf_counter() - wall0
    barrier(world, device)
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_s = sum(times_ms) / 1000.0
    max_s = all_max(kernel_s, world, device)
    clk = clocks.summary()
    code, flags = plan.status(stream)
    if code != smla.SMLA_OK:
        raise RuntimeError(f"device status {code} flags {flags} in the timed region")
    stats = step_stats(times_ms)

    # ------------------------------------------------ back-to-back launches (warm L2), secondary
    warm = None
    if not args.no_warm:
        n_warm = max(3, min(args.steps, 50))
        ew0 = torch.cuda.Event(enable_timing=True)
        ew1 = torch.cuda.Event(enable_timing=True)
        step()
        ew0.record(stream)
        for _ in range(n_warm):
            step()
        ew1.record(stream)
        torch.cuda.synchronize(device)
        warm_s = all_max(ew0.elapsed_time(ew1) / 1000.0, world, device)
        warm = {"ms_per_launch": 1000 * warm_s / n_warm, "launches": n_warm,
                "value": world * pairs * n_warm / warm_s, "unit": UNIT,
                "note": "back to back, no L2 flush between launches (outside the timed region)"}

    # ------------------------------------------------ end to end through the host API
    e2e = None
    if not args.no_e2e:
        pin = {k: (None if v is None else v.pin_memory()) for k, v in host.items()}
        pin["out"] = torch.empty(plan.output_shape, dtype=torch.float32).pin_memory()
        dev2 = dict(dev)
        dev2["out"] = out
        e_steps = max(3, min(args.steps, args.e2e_steps))
        for _ in range(2):
            plan.run_from_host(pin, dev2, stream=stream)
        torch.cuda.synchronize(device)
        barrier(world, device)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(e_steps):
            plan.run_from_host(pin, dev2, stream=stream)
        ev1.record(stream)
        torch.cuda.synchronize(device)
        e2e_s = all_max(ev0.elapsed_time(ev1) / 1000.0, world, device)
        sizes = plan.io_sizes
        h2d = sizes.q_bytes + sizes.k_bytes + sizes.lse_bytes + sizes.indices_bytes + sizes.topk_length_bytes
        e2e = {"value": world * pairs * e_steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(sizes.out_bytes), "steps": e_steps,
               "ms_per_step": 1000 * e2e_s / e_steps}

    hbm_gbs, bf16_tf, src = load_peaks()

    # ------------------------------------------------ the forward-LSE modes (outside the timed region)
    lse_modes = None
    if not args.no_lse_modes:
        lse_buf = torch.empty(plan.lse_shape, dtype=torch.float32, device=device)
        extra = dict(sparse_indices=dev["indices"], topk_length=dev["topk_length"], stream=stream)
        modes = {
            "lse_forward": (lambda: plan.softmax_lse(dev["q"], dev["k"], lse_out=lse_buf, **extra), 1),
            "lse_then_l1norm_fused": (lambda: plan.run_fused_lse(dev["q"], dev["k"], out=out, lse_out=lse_buf,
                                                                 **extra), 2),
        }
        lse_modes = {}
        for mname, (fn, passes) in modes.items():
            for _ in range(3):
                flush()
                fn()
            torch.cuda.synchronize(device)
            ms_list = timed_launches(fn, args.lse_steps, stream, flush)
            code, flags = plan.status(stream)
            if code != smla.SMLA_OK:
                raise RuntimeError(f"device status {code} flags {flags} in mode {mname}")
            st = step_stats(ms_list)
            ms = all_max(st["median"], world, device)
            tf = passes * flops / (ms / 1000.0) / 1e12
            lse_modes[mname] = {"ms_per_launch": st, "pairs_per_s": world * pairs / (ms / 1000.0), "tflops": tf,
                                "mma_passes": passes,
                                "roofline_tensor": {"achieved": tf, "peak": bf16_tf, "unit": "TFLOP/s",
                                                    "frac": tf / bf16_tf, "peak_source": src}}

    # ------------------------------------------------ the other configurations (outside the timed region)
    others = None
    if world == 1 and not args.no_other_configs and args.seq_len is None:
        del host
        others = {}
        for n in (1, 2, 3, 4, 5):
            if n != args.config:
                others[str(n)] = other_config_line(smla, n, args.other_steps, device, stream, flush,
                                                   gpu_uuid if gpu_uuid else local)

    if rank != 0:
        return 0

    # ------------------------------------------------ CPU oracle baseline
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        threads = host_threads()
        r = cpu_oracle_run(args.config, 1, 1, args.cpu_seconds, threads, seq_len=args.seq_len)
        n_rows, c_pairs, c_secs = r["steps"][0]
        cpu = {"value": c_pairs / c_secs, "unit": UNIT, "cores": threads, "kind": "oracle", "cpu": cpu_model(),
               "sample": f"{n_rows} random rows of {name} in {c_secs:.1f}s (fp64 numpy, BLAS threads={threads})"}

    per_launch_s = kernel_s / args.steps
    l1_kernel = l1_kernel_name(plan)
    traffic = profiled_traffic(name, l1_kernel)
    t_tc = flops / (bf16_tf * 1e12)
    line = {
        "metric": METRIC, "value": world * pairs * args.steps / max_s, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * max_s / args.steps,
        "step_ms": stats,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded numpy; q,k ~ N(0,1) rounded to the dtype; LSE = its expected value "
                "ln(kept slots) + scale^2 |q_g|^2 / 2, which leaves the work unchanged)",
        "config": {"workload": name, "layout": w.layout, "B": w.batch, "S1": w.max_seqlen_q,
                   "S2": int(w.k_bits.shape[1]) if w.layout == "BSND" else None, "N1": w.G, "D": w.head_dim,
                   "topk": w.topk, "mask_mode": w.mask_mode, "pairs_per_step": pairs,
                   "flops_per_step": flops, "algorithmic_bytes_per_step": alg_bytes,
                   "compulsory_bytes_per_step": comp_bytes,
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed before every timed launch: 512 MB written, then 256 MB read (write-backs "
                         "of the flush land before the launch)"},
        "tflops": world * flops * args.steps / max_s / 1e12,
        "roofline": dict(roofline_block(flops, comp_bytes, per_launch_s, hbm_gbs, bf16_tf, src, traffic),
                         kernel=l1_kernel),
        "roofline_tensor": {"achieved": flops / per_launch_s / 1e12, "peak": bf16_tf, "unit": "TFLOP/s",
                            "frac": flops / per_launch_s / 1e12 / bf16_tf, "peak_source": src},
        "gathered_bytes_roofline": gathered_bytes_block(alg_bytes, per_launch_s, hbm_gbs, t_tc),
        "clocks": clk,
        "gpu_launches": args.steps,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "lse_modes": lse_modes,
        "warm_back_to_back": warm,
        "other_configs": others,
        "wall_s_timed_region": wall,
        "plan": {k: v for k, v in plan.info.as_dict().items() if k in ("num_ctas", "stages", "mma_n",
                                                                        "smem_bytes", "max_cta_cost",
                                                                        "mean_cta_cost", "mma_issuers",
                                                                        "cta_pairs", "split_tiles", "split_items")},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=3.0,
                    help="reference arm: CPU seconds per step at most")
    ap.add_argument("--ref-total-seconds", type=float, default=120.0,
                    help="reference arm: CPU seconds over all timed steps at most")
    ap.add_argument("--no-lse-modes", action="store_true",
                    help="skip timing the forward-LSE and fused LSE+L1-norm launches")
    ap.add_argument("--lse-steps", type=int, default=50)
    ap.add_argument("--no-warm", action="store_true", help="skip the back-to-back (warm L2) timing")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip timing the other four configurations after the headline")
    ap.add_argument("--other-steps", type=int, default=20, help="timed launches per other configuration")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="configs 3 and 5 only: a shorter S1 = S2 of the same workload (small profiling case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
