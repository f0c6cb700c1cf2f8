#!/usr/bin/env python3
"""Benchmark of the fused attention forward on one or more GPUs.

Default workload (the headline line): score_mod MHA forward, B=4, H=16,
L=2048, d=64, bf16 N(0,1) inputs; one step runs the three variants
(a) ALiBi with slopes 2^(-8h/H), (b) tanh softcap 30, (c) causal sliding
window 256 over the same batch.  value = unmasked-tile TFLOP/s of the whole
step (see flashattention_attn_fwd_gb300/flops.py).  Inputs rotate over three
device-resident sets (201 MB > the 129 MB L2), so every step reads cold data.

Also reported on the same line: per-workload results for every variant
configuration ("variants"), the roofline of the dominant kernel, an
end-to-end figure with pinned host buffers and host<->device copies in the
timed region ("e2e"), the SM clocks sampled during the timed region, and
the fp64 CPU oracle timed on a bounded sample ("cpu_baseline").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torch.distributed.run: every rank runs the same workload on
its own GPU (independent replicas, no data exchange); timing is the max
over ranks and value the total over ranks.  ``--impl reference`` times the
fp64 CPU oracle (the only reference implementation of this method) on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from flashattention_attn_fwd_gb300 import flops as F  # noqa: E402
from flashattention_attn_fwd_gb300 import synth  # noqa: E402

METRIC = "attention fwd TFLOP/s (unmasked FLOPs) per variant and % of GB300 roofline"
UNIT = "TFLOP/s"
B, H, L, D = 4, 16, 2048, 64
HEADLINE = [
    ("alibi", dict(score_mod="alibi")),
    ("softcap", dict(score_mod="softcap", softcap=30.0)),
    ("window", dict(mask="window", window=256)),
]


# --------------------------------------------------------------------- peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm=float(pk["hbm_gbs"]), bf16=float(pk["bf16_tflops"]),
                    bf16_sustained=float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# -------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock, power and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.lines: list[str] = []
        self.proc = None
        self.thread = None

    def start(self):
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ workloads
def headline_inputs(seed, device):
    q, k, v = synth.attn_inputs(B, H, H, L, D, seed=seed)
    return [t.to(device) for t in (q, k, v)]


def headline_counts():
    out = {}
    for name, kw in HEADLINE:
        mk = {k: v for k, v in kw.items() if k in ("mask", "window")}
        out[name] = F.attn_counts(B, H, H, L, D, **mk)
    return out


def make_calls(api, bufs, slopes):
    q, k, v, outs = bufs
    calls = []
    for idx, (name, kw) in enumerate(HEADLINE):
        kw2 = dict(kw)
        if name == "alibi":
            kw2["alibi_slopes"] = slopes
        o, lse = outs[idx]
        calls.append((name, lambda kw2=kw2, o=o, lse=lse: api.attn_fwd(q, k, v, out=o, lse=lse, **kw2)))
    return calls


# Each kernel family is built from every source file except the ones only
# another family uses, so a change to (say) the backward leaves the forward
# kernels' counters valid.
KERNEL_FAMILY_EXCLUDES = {"forward": ("bwd.", "decode."), "backward": ("decode.",), "decode": ("bwd.",)}
TRAFFIC_FAMILY = {"decode": "decode", "backward": "backward", "backward_d128": "backward",
                  "diffattn_backward": "backward"}  # every other entry: forward


def kernel_source_hash(family="forward"):
    """Hash of the sources one kernel family is compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "flashattention_attn_fwd_gb300", "csrc")
    skip = KERNEL_FAMILY_EXCLUDES[family]
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh", ".h")) or f.startswith(skip):
            continue
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of that kernel's family; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            tr = json.load(f)
    except (OSError, ValueError):
        return None
    fam = TRAFFIC_FAMILY.get(kernel_key, "forward")
    if tr.get("source_hashes", {}).get(fam) != kernel_source_hash(fam):
        return None
    ent = tr.get("kernels", {}).get(kernel_key)
    return None if ent is None else ent.get("dram_bytes_per_launch")


# ----------------------------------------------------------- variant configs
def variant_configs():
    """Every workload configuration as (name, builder) pairs; builders return
    (callable, tile_flops, exact_flops, bytes, l2_note)."""
    from flashattention_attn_fwd_gb300 import api

    dev = torch.device("cuda")

    def attn(name, Bb, Hq, Hkv, Ll, d, nsets, seed, **kw):
        def build():
            sets = []
            offs = synth.doc_offsets(Bb, Ll, 8, seed=seed) if kw.get("mask") == "document" else None
            for s in range(nsets):
                q, k, v = (t.to(dev) for t in synth.attn_inputs(Bb, Hq, Hkv, Ll, d, seed=seed + s))
                sets.append((q, k, v, torch.empty_like(q), torch.empty(Bb, Hq, Ll, device=dev)))
            gkw = dict(kw)
            if offs is not None:
                gkw["doc_offsets"] = offs.to(dev)
            if kw.get("score_mod") == "alibi":
                gkw["alibi_slopes"] = synth.alibi_slopes(Hq).to(dev)
            mk = {a: b for a, b in kw.items() if a in ("mask", "window", "prefix", "doc_causal")}
            tf, ef, by = F.attn_counts(Bb, Hq, Hkv, Ll, d, doc_offsets=None if offs is None else offs.numpy(), **mk)
            it = [0]

            def call():
                q, k, v, o, lse = sets[it[0] % nsets]
                it[0] += 1
                api.attn_fwd(q, k, v, out=o, lse=lse, **gkw)
            return call, tf, ef, by, f"{nsets} rotating input sets"
        return name, build

    def diff():
        def build():
            t = [x.to(dev) for x in synth.diff_inputs(4, 16, 4096, seed=40)]
            o = torch.empty(4, 16, 4096, 128, device=dev, dtype=torch.bfloat16)
            lse = torch.empty(2, 4, 16, 4096, device=dev)
            tf, ef, by = F.diff_counts(4, 16, 4096)

            def call():
                api.diffattn_fwd(*t, 0.8, out=o, lse=lse)
            return call, tf, ef, by, "1 input set (271 MB > L2)"
        return "4 diffattn B4 H16 L4096 causal lambda0.8", build

    def evo_col():
        def build():
            sets = []
            for s_ in range(2):
                e = [x.to(dev) for x in synth.evo_col_inputs(1, 128, 256, 8, d=32, seed=70 + s_)]
                sets.append((e, torch.empty_like(e[0]), torch.empty(1, 8, 256, 128, device=dev)))
            tf, ef, by = F.evo_col_counts(1, 128, 256, 8)
            it = [0]

            def call():
                e, o, lse = sets[it[0] % 2]
                it[0] += 1
                api.evoformer_col_gated_attn_fwd(*e, out=o, lse=lse)
            return call, tf, ef, by, "2 rotating input sets (170 MB > L2)"
        return "5col evoformer-column Ns128 Nr256 H8 d32", build

    def decode():
        def build():
            q, k, v, kv_len = synth.decode_inputs(16, 32, 8, 1, 8192, 64, seed=61)
            q, k, v, kv_len = q.to(dev), k.to(dev), v.to(dev), kv_len.to(dev)
            o = torch.empty_like(q)
            lse = torch.empty(16, 32, 1, device=dev)
            tf, ef, by = F.decode_counts(16, 32, 8, 1, 64, kv_len.cpu().numpy())
            from flashattention_attn_fwd_gb300 import _lib
            import ctypes
            desc = _lib.new_desc()
            desc.B, desc.Hq, desc.Hkv, desc.Lq, desc.Lk, desc.d, desc.dv = 16, 32, 8, 1, 8192, 64, 64
            need = int(_lib.lib().fl_attn_decode_workspace_size(ctypes.byref(desc)))
            ws = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)

            def call():
                api.attn_decode_fwd(q, k, v, kv_len, out=o, lse=lse, workspace=ws)
            return call, tf, ef, by, "1 input set (269 MB cache > L2)"
        return "6 decode B16 Hq32 Hkv8 Lq1 cache8192 d64 mixed-lengths", build

    def bwd(name, Bb, Hh, Ll, d, seed, **kw):
        def build():
            q, k, v = (t.to(dev) for t in synth.attn_inputs(Bb, Hh, Hh, Ll, d, seed=seed))
            dout = synth.randn_bf16((Bb, Hh, Ll, d), synth.generator(seed + 1)).to(dev)
            out, lse = api.attn_fwd(q, k, v, **kw)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws = torch.empty(Bb * Hh * Ll * (d + 2) * 4, device=dev, dtype=torch.uint8)
            tf, ef, by = F.bwd_counts(Bb, Hh, Hh, Ll, d, **kw)

            def call():
                api.attn_bwd(q, k, v, out, dout, lse, dq=dq, dk=dk, dv=dv, workspace=ws, **kw)
            mb = (8 * q.numel() * 2 + q.numel() * 4) / 1e6
            return call, tf, ef, by, f"1 input set ({mb:.0f} MB of inputs, outputs and dq accumulator)"
        return name, build

    def diff_bwd():
        def build():
            q1, k1, q2, k2, v = (t.to(dev) for t in synth.diff_inputs(4, 16, 4096, seed=40))
            dout = synth.randn_bf16((4, 16, 4096, 128), synth.generator(41)).to(dev)
            grads = [torch.empty_like(t) for t in (q1, k1, q2, k2, v)]
            ws = torch.empty(4 * 16 * 4096 * 784, device=dev, dtype=torch.uint8)
            tf, ef, by = F.diff_bwd_counts(4, 16, 4096)

            def call():
                api.diffattn_bwd(q1, k1, q2, k2, v, dout, 0.8, causal=True, dq1=grads[0], dk1=grads[1],
                                 dq2=grads[2], dk2=grads[3], dv=grads[4], workspace=ws)
            return call, tf, ef, by, "1 input set (268 MB of inputs, 201 MB of gradients, 206 MB workspace)"
        return "4b diffattn backward B4 H16 L4096 causal lambda0.8", build

    def evo():
        def build():
            sets = []
            for s in range(2):
                e = [x.to(dev) for x in synth.evo_inputs(1, 128, 256, 8, d=32, seed=50 + s)]
                sets.append((e, torch.empty_like(e[0]), torch.empty(1, 128, 8, 256, device=dev)))
            tf, ef, by = F.evo_counts(1, 128, 256, 8)
            it = [0]

            def call():
                e, o, lse = sets[it[0] % 2]
                it[0] += 1
                api.evoformer_gated_attn_fwd(*e, out=o, lse=lse)
            return call, tf, ef, by, "2 rotating input sets (174 MB > L2)"
        return "5 evoformer Ns128 Nr256 H8 d32", build

    return [
        attn("1 causal B1 H2 L256 d64", 1, 2, 2, 256, 64, 1, 1, mask="causal"),
        attn("2a alibi B4 H16 L2048 d64", 4, 16, 16, 2048, 64, 3, 2, score_mod="alibi"),
        attn("2b softcap30 B4 H16 L2048 d64", 4, 16, 16, 2048, 64, 3, 5, score_mod="softcap", softcap=30.0),
        attn("2c window256 B4 H16 L2048 d64", 4, 16, 16, 2048, 64, 3, 8, mask="window", window=256),
        attn("3a gqa32/8 doc8 B2 L8192 d64", 2, 32, 8, 8192, 64, 2, 11, mask="document"),
        attn("3b gqa32/8 prefix1024 B2 L8192 d64", 2, 32, 8, 8192, 64, 2, 13, mask="prefix_lm", prefix=1024),
        diff(),
        diff_bwd(),
        evo(),
        evo_col(),
        decode(),
        bwd("7 backward B4 H16 L2048 d64 causal", 4, 16, 2048, 64, 90, mask="causal"),
        attn("8 d128 causal B2 H16 L4096 d128", 2, 16, 16, 4096, 128, 2, 70, mask="causal"),
        bwd("9 backward d128 B2 H16 L4096 causal", 2, 16, 4096, 128, 92, mask="causal"),
    ]


def time_call(call, reps, warmup=3):
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    return statistics.median(ms), ms


def run_variants(peaks):
    res = {}
    for name, build in variant_configs():
        call, tf, ef, by, note = build()
        med, _ = time_call(call, reps=20)
        from flashattention_attn_fwd_gb300 import sync_status
        sync_status()
        t_roof, bound = F.roofline_time(tf, by, peaks["bf16"], peaks["hbm"])
        res[name] = {
            "ms": round(med, 4),
            "tflops_tile": round(tf / (med * 1e-3) / 1e12, 2),
            "tflops_exact": round(ef / (med * 1e-3) / 1e12, 2),
            "gbs": round(by / (med * 1e-3) / 1e9, 1),
            "bound": bound,
            "roofline_frac": round(t_roof / (med * 1e-3), 4),
            "l2": note,
        }
        del call
        torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ CPU oracle
_INPUT_CACHE = {}


def _oracle_head(args):
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import oracle
    b, h, name, seed = args
    if seed not in _INPUT_CACHE:
        _INPUT_CACHE[seed] = synth.attn_inputs(B, H, H, L, D, seed=seed)
    q, k, v = _INPUT_CACHE[seed]
    kw = dict(HEADLINE)[name]
    okw = {a: bb for a, bb in kw.items()}
    if name == "alibi":
        okw["slopes"] = synth.alibi_slopes(H)[h:h + 1]
    oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], **okw)
    return 1


def cpu_model() -> str:
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5)
        for ln in r.stdout.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part", "hardware")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def git_sha():
    try:
        r = subprocess.run(["git", "-C", ROOT, "rev-parse", "--short=12", "HEAD"], capture_output=True, text=True,
                           timeout=5)
        return r.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        return None


def oracle_sample(n_heads: int, seed: int = 0):
    """Run the fp64 oracle on n_heads (b, h) heads of each headline variant
    with a spawn process pool; returns (TFLOP/s, wall s, workers, desc)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    workers = max(1, min(cores, 16, n_heads * len(HEADLINE)))
    jobs = [(i // H % B, i % H, name, seed) for name, _ in HEADLINE for i in range(n_heads)]
    cnt = headline_counts()
    flops = sum(cnt[name][0] / (B * H) * n_heads for name, _ in HEADLINE)
    env_old = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env_old:
        os.environ[k] = "1"
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        pool.map(_oracle_head, jobs[:workers])  # warm the workers (imports, input generation)
        t0 = time.perf_counter()
        pool.map(_oracle_head, jobs)
        wall = time.perf_counter() - t0
    for k, v in env_old.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v
    what = "the whole headline step" if n_heads == B * H else f"{n_heads} of the {B * H} (b,h) heads"
    desc = (f"fp64 oracle, {what} (3 variants of B{B} H{H} L{L} d{D}), "
            f"{workers} worker processes x 1 BLAS thread")
    return flops / wall / 1e12, wall, workers, desc


def run_profile(args):
    """A few launches of one workload (for ncu): warmup + 3 timed-free calls."""
    torch.cuda.set_device(0)
    from flashattention_attn_fwd_gb300 import sync_status
    for name, build in variant_configs():
        if name.startswith(args.profile):
            call = build()[0]
            for _ in range(args.warmup + 3):
                call()
            sync_status()
            print(f"profiled {name}: {args.warmup} warm-up + 3 launches")
            return 0
    raise SystemExit(f"no workload named {args.profile!r}")


# ------------------------------------------------------------------- main
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    n_heads = B * H  # each step: the whole headline step
    for _ in range(args.warmup):
        oracle_sample(n_heads)
    vals, walls = [], []
    for _ in range(args.steps):
        v, w, workers, desc = oracle_sample(n_heads)
        vals.append(v)
        walls.append(w)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(walls), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"score_mod MHA fwd B={B} H={H} L={L} d={D}: ALiBi, softcap 30, "
                               "causal window 256", "sample_per_step": f"{n_heads} (b,h) heads x 3 variants"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
                         "workers": workers, "cpu_model": cpu_model(), "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", default=None,
                    help="run --warmup + 3 launches of the workload whose name starts with this "
                         "prefix (e.g. 2b, 5) and exit; for ncu captures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from flashattention_attn_fwd_gb300 import api, sync_status
    peaks = load_peaks()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # ---- headline: three variants per step over rotating input sets
    nsets = 3
    slopes = synth.alibi_slopes(H).to(dev)
    sets = []
    for s in range(nsets):
        q, k, v = headline_inputs(100 + s, dev)
        outs = [(torch.empty_like(q), torch.empty(B, H, L, device=dev)) for _ in HEADLINE]
        sets.append(make_calls(api, (q, k, v, outs), slopes))
    counts = headline_counts()
    step_flops = sum(c[0] for c in counts.values())
    step_exact = sum(c[1] for c in counts.values())

    def step(i):
        for _, c in sets[i % nsets]:
            c()

    for i in range(args.warmup):
        step(i)
    sync_status()
    K = args.steps
    ev = {name: [] for name, _ in HEADLINE}
    sampler = ClockSampler(local)
    barrier()
    sampler.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(K):
        for name, c in sets[i % nsets]:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            c()
            b.record()
            ev[name].append((a, b))
    t1.record()
    barrier()
    clocks = sampler.stop()
    sync_status()
    total_ms = t0.elapsed_time(t1)
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_per_step = total_ms / K
    value = step_flops * K * world / (total_ms * 1e-3) / 1e12
    per = {name: statistics.mean(a.elapsed_time(b) for a, b in ev[name]) for name in ev}
    dom = max(per, key=lambda n: per[n])
    tf, ef, by = counts[dom]
    t_roof, bound = F.roofline_time(tf, by, peaks["bf16"], peaks["hbm"])
    dur = per[dom] * 1e-3
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": round(tf / dur / 1e12, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": round(tf / dur / 1e12 / peaks["bf16"], 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(by / dur / 1e9, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(by / dur / 1e9 / peaks["hbm"], 4)}
    roof["traffic"] = ncu_traffic(dom)
    roof["kernel"] = f"fused_attn_fwd_kernel<64,64,ATTN,{dom}>"
    roof["peak_source"] = f"{peaks['source']} (burst bf16 / copy HBM)"
    roof["per_kernel_ms"] = {n: round(v, 4) for n, v in per.items()}

    # ---- end to end: pinned host buffers, copies inside the timed region.
    # Every step copies its inputs in from pinned host memory, runs the three
    # calls and copies every result (out and lse) back.  Steps overlap on
    # three streams, as a serving loop would: step k's inputs come in (copy
    # stream) while step k-1's kernels run (compute stream) and its results
    # go out (a second copy stream, each result as soon as its kernel is
    # done).  The copies then bound the step: about 100 MB cross the host
    # link per step.  Device inputs and results are double-buffered; events order
    # each buffer's reuse.  The timed region runs from before the first copy
    # of the first timed step to after the last copy of the last one.
    hq, hk, hv = (t.cpu().pin_memory() for t in headline_inputs(200, "cpu"))
    NBUF = 2
    din = [[torch.empty_like(t, device=dev) for t in (hq, hk, hv)] for _ in range(NBUF)]
    # the three calls' LSEs are slices of one buffer, read back in one copy
    dlse = [torch.empty(len(HEADLINE), B, H, L, device=dev) for _ in range(NBUF)]
    douts = [[(torch.empty(hq.shape, dtype=torch.bfloat16, device=dev), dlse[i][j]) for j in range(len(HEADLINE))]
             for i in range(NBUF)]
    houts = [torch.empty(hq.shape, dtype=torch.bfloat16).pin_memory() for _ in HEADLINE]
    hlse = torch.empty(len(HEADLINE), B, H, L).pin_memory()
    ecalls = [make_calls(api, (din[i][0], din[i][1], din[i][2], douts[i]), slopes) for i in range(NBUF)]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(NBUF)]             # inputs of buffer i landed
    ev_used = [torch.cuda.Event() for _ in range(NBUF)]           # kernels done with inputs i
    ev_kern = [[torch.cuda.Event() for _ in HEADLINE] for _ in range(NBUF)]
    ev_out = [torch.cuda.Event() for _ in range(NBUF)]            # results i copied out
    started = [False] * NBUF

    def e2e_step(k):
        i = k % NBUF
        if started[i]:
            s_in.wait_event(ev_used[i])
        with torch.cuda.stream(s_in):
            din[i][0].copy_(hq, non_blocking=True)
            din[i][1].copy_(hk, non_blocking=True)
            din[i][2].copy_(hv, non_blocking=True)
            ev_in[i].record(s_in)
        comp.wait_event(ev_in[i])
        if started[i]:
            comp.wait_event(ev_out[i])
        for j, (_, c) in enumerate(ecalls[i]):
            c()
            ev_kern[i][j].record(comp)
        ev_used[i].record(comp)
        with torch.cuda.stream(s_out):
            for j, ((o, _), ho) in enumerate(zip(douts[i], houts)):
                s_out.wait_event(ev_kern[i][j])
                ho.copy_(o, non_blocking=True)
            hlse.copy_(dlse[i], non_blocking=True)
            ev_out[i].record(s_out)
        started[i] = True

    def e2e_drain():
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)

    for w in range(args.warmup):
        e2e_step(w)
    e2e_drain()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    s_in.wait_stream(comp)
    s_out.wait_stream(comp)
    for k in range(K):
        e2e_step(args.warmup + k)
    e2e_drain()
    e1.record(comp)
    barrier()
    sync_status()
    e2e_ms = e0.elapsed_time(e1)
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = float(tt.item())
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = sum(o.numel() * o.element_size() for o in houts) + hlse.numel() * hlse.element_size()
    e2e = {"value": round(step_flops * K * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_ms / K, 4)}

    variants = None if args.no_variants else run_variants(peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, wall, workers, desc = oracle_sample(n_heads=B * H)
        cpu = {"value": round(v, 6), "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "workers": workers,
               "cpu_model": cpu_model(), "kind": "oracle", "sample": desc, "wall_s": round(wall, 2),
               "cpu_s": round(wall * workers, 1)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"score_mod MHA fwd B={B} H={H} L={L} d={D}: ALiBi slopes 2^(-8h/H), "
                                   "tanh softcap 30, causal sliding window 256 (one call each per step)",
                       "B": B, "H": H, "L": L, "d": D, "parallelism": f"replicas x{world}",
                       "l2": "3 rotating device input sets (201 MB > 129 MB L2)",
                       "flops": "unmasked 128x128 tiles", "exact_pair_tflops": round(
                           step_exact * K * world / (total_ms * 1e-3) / 1e12, 3)},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": K * len(HEADLINE),
            "clocks": clocks,
            "variants": variants,
            "git_sha": git_sha(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
