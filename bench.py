"""Benchmark: the 27B-shaped Q4 verify pass at K+1 = 4 on one GB300 (replicas on N GPUs).

One step = one whole verify pass: 64 layers x 4 fused 4-bit verify-linear launches over the 4
window columns, the lm_head (5120 x 151936) with the production sampler over the 4 positions, and
the acceptance of the 3 drafts.  Inputs are synthetic (seeded), resident in HBM; the 11.9 GB of
weights per step exceed the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl svd|reference]

Prints one JSON line on rank 0.  --impl reference times the fp64 CPU oracle on the host cores,
one whole verify pass per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "27B-shape Q4 verify passes/s at K+1=4"
UNIT = "passes/s"
WORKLOAD = ("27B-shaped dense Q4 verify pass, K+1=4: 64 layers x (qkv 5120x7168, o 5120x5120, "
            "gate|up 5120x34816, down 17408x5120) + lm_head 5120x151936 + sampler "
            "(T 0.6, top-p 0.95, min-p 0.05) + acceptance of 3 drafts")
FALLBACK_HBM_GBS = 6800.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if key in d:
                return float(d[key]), "measured"
    except Exception:
        pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_sha16() -> str:
    """First 16 hex digits of the sha256 of the verify-linear translation unit's sources
    (verify_linear.cu followed by the headers it includes from the package)."""
    d = os.path.join(ROOT, "speculative_decoding_verify_06_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("verify_linear.cu", "verify_linear_tc.cuh", "svd_common.cuh"):
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def kernel_traffic(summary="vl_stream_kernel_27b_stack_c4.txt"):
    """DRAM traffic per launch of the stack's verify-linear kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    prof = os.path.join(ROOT, "profiles", summary)
    try:
        sha = kernel_source_sha16()
        txt = open(prof).read()
        m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
        m_tr = re.search(r"dram_bytes_per_stack_launch_avg:\s*([0-9.eE+]+)", txt)
        if m_sha and m_tr and m_sha.group(1) == sha:
            return float(m_tr.group(1))
    except Exception:
        pass
    return None


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over the ranks of the default process group (the slowest replica's time),
    or x itself when there is no group."""
    import torch
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()) or td.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def replica_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job rate of `world` replicas that each processed `units_per_rank` units, timed by
    the slowest rank (units per second)."""
    return world * units_per_rank / (ms_max / 1000.0)


def percentiles(xs):
    """median, p10 and p90 of a list of per-step times."""
    ys = sorted(xs)
    def pct(q):
        if len(ys) == 1:
            return ys[0]
        i = q * (len(ys) - 1)
        lo = int(i)
        hi = min(lo + 1, len(ys) - 1)
        return ys[lo] + (ys[hi] - ys[lo]) * (i - lo)
    return {"median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9)}


def _cpu_model() -> str:
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part", "hardware")):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


class OracleSample:
    """The fp64 oracle timed on the host, one step = one whole verify pass at C = 4: the four
    fused GEMMs of a layer (every row) 64 times -- one layer's matrices stand for all 64, the
    same arithmetic and the same bytes streamed from host memory per layer -- then the whole
    lm_head (5120 x 151936), the sampler over the 4 target and 3 drafter positions, and the
    acceptance of one window of 3 drafts.  With `layers` < 64 a step is that many layers and the
    lm_head share of the same fraction (a bounded sample: passes_per_s scales it, and `fraction`
    says by how much)."""

    def __init__(self, layers: int = 64, threads: int = 0):
        import numpy as np

        import oracle
        from speculative_decoding_verify_06_gb300 import synth
        self.np, self.oracle, self.synth = np, oracle, synth
        self.threads = threads or oracle.max_threads()
        self.layers = layers
        self.fraction = layers / synth.LAYERS
        C = 4
        self.mats = [synth.qweight(o, i, seed=1000 + g) for g, (i, o) in enumerate(synth.LAYER_GEMMS)]
        self.xs = [synth.activations(C, i, seed=2000 + g) for g, (i, o) in enumerate(synth.LAYER_GEMMS)]
        head_rows = max(16, int(round(synth.VOCAB * self.fraction)))
        self.head = synth.qweight(head_rows, synth.HIDDEN, seed=1999)
        self.hx = synth.activations(C, synth.HIDDEN, seed=2999)
        self.weights = (layers * sum(i * o for i, o in synth.LAYER_GEMMS) + head_rows * synth.HIDDEN)

    def step(self) -> float:
        np, oracle = self.np, self.oracle
        f32 = np.float32
        t0 = time.perf_counter()
        for _ in range(self.layers):
            for (c, s), x in zip(self.mats, self.xs):
                oracle.verify_linear(c, s, x, nthreads=self.threads)
        y, _ = oracle.verify_linear(self.head[0], self.head[1], self.hx, nthreads=self.threads)
        lg = y.astype(f32)
        p, *_ = oracle.sampler(lg, f32(0.6), f32(0.95), f32(0.05), nthreads=self.threads)
        q, *_ = oracle.sampler(self.synth.perturb(lg[:3], 1.205, 5), f32(0.6), f32(0.95), f32(0.05),
                               nthreads=self.threads)
        d = self.synth.draw_from(q, 6).reshape(1, 3)
        oracle.accept(p.astype(f32), d, q=q.astype(f32), seed=1, nthreads=self.threads)
        return time.perf_counter() - t0

    def passes_per_s(self, step_times) -> float:
        return self.fraction / statistics.mean(step_times)

    def describe(self, n: int) -> str:
        what = ("one whole pass" if self.layers == self.synth.LAYERS else
                f"{self.layers} of the 64 layers and the same share of the lm_head rows, scaled by "
                f"{1 / self.fraction:g} to a pass")
        return (f"{n} step(s), each {what} ({self.weights / 1e9:.2f}G weights) at C=4 in fp64: "
                f"the 4 fused GEMMs of one layer's full-size matrices per layer, lm_head, sampler "
                f"(4 + 3 rows of 151936), acceptance of one window")


def lm_head_oracle_windows(n_windows: int = 16, threads: int = 0):
    """The lm_head + sampler workload on the host: n_windows windows, each the 5120 x 151936
    lm_head over K+1 = 6 columns and the sampler over the 6 rows, in fp64 (windows per second)."""
    import numpy as np

    import oracle
    from speculative_decoding_verify_06_gb300 import synth
    threads = threads or oracle.max_threads()
    codes, scales = synth.qweight(synth.VOCAB, synth.HIDDEN, seed=4999)
    f32 = np.float32
    t0 = time.perf_counter()
    for w in range(n_windows):
        x = synth.activations(6, synth.HIDDEN, seed=5000 + w)
        y, _ = oracle.verify_linear(codes, scales, x, nthreads=threads)
        oracle.sampler(y.astype(f32), f32(0.6), f32(0.95), f32(0.05), nthreads=threads)
    dt = time.perf_counter() - t0
    return {"value": n_windows / dt, "unit": "windows/s", "cores": threads, "kind": "oracle",
            "seconds": dt, "sample": f"{n_windows} whole windows (lm_head 5120 x 151936 at C = 6 "
                                     f"+ sampler over 6 rows), fp64"}


REF_BUDGET_S = 240.0  # host seconds the reference arm may take, warm-up included


def ref_sample_layers(t_pass: float, n_steps: int, budget: float = REF_BUDGET_S,
                      layers: int = 64) -> int:
    """Layers per step so that n_steps more steps fit in what is left of the budget after the
    first whole pass of t_pass seconds (all of them while whole passes fit; at least one)."""
    left = budget - t_pass
    if n_steps <= 0 or n_steps * t_pass <= left:
        return layers
    return max(1, min(layers, int(layers * left / (n_steps * t_pass))))


def run_reference(args, rank):
    """The oracle as the reference arm: one whole pass per step while (steps + warmup) whole
    passes fit in REF_BUDGET_S, else each step a bounded sample of the pass (a share of the
    layers and of the lm_head rows, sized from the first warm-up pass); ms_per_step is the time of
    the work each step ran, and the value scales it to passes/s."""
    if rank != 0:
        return
    smp = OracleSample()  # one whole pass per step
    t_first = smp.step()  # the first warm-up step, which also sizes the others
    layers = ref_sample_layers(t_first, args.warmup - 1 + args.steps)
    if layers < 64:
        smp = OracleSample(layers=layers)
    for _ in range(args.warmup - 1):
        smp.step()
    times = [smp.step() for _ in range(args.steps)]
    v = smp.passes_per_s(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "C": 4, "oracle": "fp64 C, OpenMP", "cpu": _cpu_model()},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": smp.threads, "kind": "oracle",
                         "sample": smp.describe(args.steps), "pass_fraction_per_step": smp.fraction,
                         "first_whole_pass_s": t_first},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _gpu_id(dev) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


SWEEP_C = (1, 2, 4, 6, 8, 16, 24, 32)


def column_sweep(vp, dev, steps, tokens_per_pass, peak):
    """The stack alone (one chain launch, same resident weights) at every window width of the
    sweep; C = 32 is the batched case of 8 sequences x 4 columns.  Widths above 16 run the
    tcgen05 kernel; "32_fragment" is C = 32 on the warp-level mma.sync kernel for comparison."""
    import torch

    from speculative_decoding_verify_06_gb300 import stack, svd
    s = torch.cuda.current_stream(dev)
    out = {}
    for C, flags, name in [(c, 0, str(c)) for c in SWEEP_C] + [(32, svd.SVD_F_FRAGMENT_MMA, "32_fragment")]:
        view = stack.ColumnsView(vp, C, seed=C, flags=flags).capture()
        for _ in range(3):
            view.launch(s)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(s)
        for _ in range(steps):
            view.launch(s)
        e1.record(s)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        gbs = view.stack_bytes() / ms / 1e6
        out[name] = {"stack_ms": ms, "passes_per_s": 1000.0 / ms, "gb_s": gbs, "frac": gbs / peak,
                     "kernel": "tcgen05" if (C > 16 and not flags) else "mma.sync"}
        del view
        torch.cuda.empty_cache()
    if "32" in out and "4" in out and tokens_per_pass:
        out["batched_8x4"] = {
            "sequences": 8,
            "verify_tokens_per_s": 8 * out["32"]["passes_per_s"] * tokens_per_pass,
            "hbm_frac_vs_c4": out["32"]["gb_s"] / out["4"]["gb_s"]}
    return out


def accept_oracle_sample(P, Q, samples, pool, n, g, dev, k=3):
    """The oracle (fp64, every host thread) deciding n windows of k drafts drawn from the same
    pool as the GPU measurement, as windows per second."""
    import numpy as np
    import torch

    import oracle
    rows = torch.randint(0, pool, (n, k + 1), generator=g, device=dev)
    pick = torch.randint(0, samples.shape[1], (n, k), generator=g, device=dev)
    draft = samples[rows[:, :k], pick].to(torch.int32).cpu().numpy()
    Ph, Qh = P.cpu().numpy(), Q.cpu().numpy()
    pr, qr = rows.cpu().numpy().astype(np.int64), rows[:, :k].contiguous().cpu().numpy().astype(np.int64)
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.accept(Ph, draft, q=Qh, p_rows=pr, q_rows=qr, seed=3, nthreads=threads)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "windows/s", "cores": threads, "kind": "oracle",
            "seconds": dt, "sample": f"{n} windows at k = {k} from the same (p, q) pool, fp64"}


ACCEPT_ALPHAS = (0.35, 0.5, 0.6, 0.7, 0.8, 0.9)


def accept_pool(dev, V, pool, alpha, g):
    """A pool of (p, q) pairs: p from Zipf(1.1)-ranked logits under a random permutation, q from
    the same logits plus tau * N(0, 1) noise, tau bisected per pair so that sum min(p, q) is
    alpha (within 1e-4 after 40 halvings)."""
    import torch
    base = -1.1 * torch.log(torch.arange(1, V + 1, device=dev, dtype=torch.float32))
    lp = base[torch.argsort(torch.rand((pool, V), generator=g, device=dev), dim=1)]
    eps = torch.randn((pool, V), generator=g, device=dev)
    P = torch.softmax(lp, dim=1)
    lo = torch.zeros(pool, device=dev)
    hi = torch.full((pool,), 64.0, device=dev)
    for _ in range(40):
        tau = 0.5 * (lo + hi)
        a = torch.minimum(P, torch.softmax(lp + tau[:, None] * eps, dim=1)).sum(1)
        lo = torch.where(a > alpha, tau, lo)
        hi = torch.where(a > alpha, hi, tau)
    Q = torch.softmax(lp + (0.5 * (lo + hi))[:, None] * eps, dim=1)
    del lp, eps
    return P.contiguous(), Q.contiguous()


def accept_throughput(dev, peak, n_windows=1_000_000, ks=(1, 3, 5), pool=256, seed=7,
                      alphas=ACCEPT_ALPHAS, oracle_windows=0):
    """svd_accept on many windows whose rows come from a pool of (p, q) pairs larger than L2
    (accept_pool), for every target acceptance alpha, a stochastic drafter (x ~ q) and a greedy
    one (x = argmax q, with the one-hot q it stands for), and k in {1, 3, 5}: every position of
    a window draws its pair independently, so acceptances are i.i.d. with the pool's mean alpha.
    Reports windows/s, the bytes the kernel must read (the residual (p - q)+ row after a
    rejection, the p row for the capping draw, the probed entries) per second against the copy
    peak, and tokens per pass against (1 - a^(k+1)) / (1 - a) at the measured mean alpha."""
    import torch

    from speculative_decoding_verify_06_gb300 import svd, synth
    V = synth.VOCAB
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    s = torch.cuda.current_stream(dev)
    out = {"pool_pairs": pool, "pool_bytes": 2 * pool * V * 4, "windows": n_windows,
           "by_alpha": {}}
    for target in alphas:
        P, Q = accept_pool(dev, V, pool, target, g)
        samples = torch.multinomial(Q, 4096, replacement=True, generator=g)  # [pool, 4096]
        am = Q.argmax(dim=1)
        Q1 = torch.zeros_like(Q)
        Q1.scatter_(1, am[:, None], 1.0)
        if oracle_windows and abs(target - 0.6) < 1e-9:
            out["cpu_baseline"] = accept_oracle_sample(P, Q, samples, pool, oracle_windows, g,
                                                       dev)
        res = {}
        for drafter, Qd in (("stochastic", Q), ("greedy", Q1)):
            alpha = float(torch.minimum(P, Qd).sum(1).mean())
            r = {"alpha": alpha}
            for k in ks:
                rows = torch.randint(0, pool, (n_windows, k + 1), generator=g, device=dev)
                q_rows = rows[:, :k].contiguous()
                if drafter == "stochastic":
                    pick = torch.randint(0, 4096, (n_windows, k), generator=g, device=dev)
                    draft = samples[q_rows, pick].to(torch.int32).contiguous()
                else:
                    draft = am[q_rows].to(torch.int32).contiguous()
                tok = torch.empty((n_windows, k + 1), dtype=torch.int32, device=dev)
                ne = torch.empty(n_windows, dtype=torch.int32, device=dev)
                st = torch.empty(n_windows, dtype=torch.int32, device=dev)

                def run(sd):
                    svd.svd_accept(P, draft, n_windows, k, V, tok, ne, st, q=Qd, p_rows=rows,
                                   q_rows=q_rows, seed=sd, stream=s)
                run(1)
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                run(2)
                e1.record(s)
                torch.cuda.synchronize(dev)
                ms = e0.elapsed_time(e1)
                bonus = int((ne == k + 1).sum())
                nbytes = (n_windows - bonus) * 8 * V + bonus * 4 * V + n_windows * 8 * k
                r[f"k{k}"] = {"ms": ms, "windows_per_s": n_windows / (ms / 1000.0),
                              "gb_s": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / peak,
                              "tokens_per_pass": float(ne.double().mean()),
                              "formula": (1 - alpha ** (k + 1)) / (1 - alpha),
                              "status_nonzero": int((st != 0).sum())}
            res[drafter] = r
        out["by_alpha"][f"{target:g}"] = res
        del P, Q, Q1, samples
        torch.cuda.empty_cache()
    return out


KV_CONTEXTS = (32768, 131072, 262144)


def kv_oracle_sample(q, kc, ks, vc, vs, n_past, C):
    """The oracle (fp64, every host thread) on one kv head of a layer's cache -- its 5 query heads
    at the window's C positions over the whole context -- as cache bytes per second."""
    import numpy as np
    import torch

    import oracle
    from speculative_decoding_verify_06_gb300 import svd, synth
    G = synth.N_Q_HEADS // synth.N_KV_HEADS
    qh = q[:, :G].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    host = [kc[:1].cpu().numpy(), ks[:1].cpu().numpy().view(np.uint16), vc[:1].cpu().numpy(),
            vs[:1].cpu().numpy().view(np.uint16)]
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.kv_attention(qh, *host, n_past, nthreads=threads)
    dt = time.perf_counter() - t0
    nbytes = -(-(n_past + C) // 16) * svd.SVD_KV_UNIT_BYTES
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": dt,
            "sample": (f"one kv head ({G} query heads x {C} window positions) over {n_past + C} "
                       f"positions, fp64; GB/s of its cache bytes")}


def kv_read(dev, peak, stack_ms, layers=64, contexts=KV_CONTEXTS, steps=10, C=4, seed=5,
            oracle_sample=False):
    """The KV-read term of a pass: svd_kv_attention once per layer (40 query heads over 8 kv heads
    of dimension 128, q8_0 keys and q4_0 values), each layer on its own cache, at the window's
    last position n_past + C = context.  The 64 layer launches (split pass + merge each) are
    recorded in one CUDA graph; all caches together exceed L2.  Reports the per-pass time, the
    cache bytes read per second against the copy peak, and the pass rate of weights plus KV read
    (this stack time plus the KV time, measured apart)."""
    import torch

    from speculative_decoding_verify_06_gb300 import svd, synth
    Hq, Hkv, D = synth.N_Q_HEADS, synth.N_KV_HEADS, synth.HEAD_DIM
    s = torch.cuda.current_stream(dev)
    out = {}
    for ctx in contexts:
        n_past = ctx - C
        nbytes = svd.svd_kv_cache_bytes(Hkv, ctx)
        kc, ks, vc, vs = synth.kv_cache_torch(Hkv, ctx, D, seed, dev)
        caches = []
        for _ in range(layers):
            cache = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            svd.svd_kv_repack(kc, ks, vc, vs, Hkv, ctx, 0, ctx, cache, ctx, stream=s)
            caches.append(cache)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        q = torch.randn((C, Hq, D), generator=g, device=dev).to(torch.bfloat16)
        if oracle_sample and "cpu_baseline" not in out:
            out["cpu_baseline"] = kv_oracle_sample(q, kc, ks, vc, vs, ctx - C, C)
        del kc, ks, vc, vs
        o = torch.empty((C, Hq, D), dtype=torch.float32, device=dev)
        ws = torch.zeros(svd.svd_kv_attention_workspace_bytes(Hq, Hkv, C), dtype=torch.uint8,
                         device=dev)
        scale = 1.0 / D ** 0.5

        def one_pass(st):
            for cache in caches:
                svd.svd_kv_attention(q, cache, ctx, Hq, Hkv, n_past, C, scale, o, ws, stream=st)
        one_pass(s)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(dev)
        with torch.cuda.stream(cs):
            graph.capture_begin()
            one_pass(cs)
            graph.capture_end()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            graph.replay()
        e1.record(s)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        read = layers * (Hkv * -(-ctx // 16) * svd.SVD_KV_UNIT_BYTES + C * Hq * D * (2 + 4))
        gbs = read / ms / 1e6
        flags = int(ws[:4].view(torch.int32).item())
        out[str(ctx)] = {"kv_ms_per_pass": ms, "per_layer_us": 1000.0 * ms / layers,
                         "kv_bytes_per_pass": read, "gb_s": gbs, "frac": gbs / peak,
                         "wait_flags": flags}
        if stack_ms:
            out[str(ctx)]["passes_per_s_weights_plus_kv"] = 1000.0 / (stack_ms + ms)
        del graph, caches, q, o, ws
        torch.cuda.empty_cache()
    out["launches_per_pass"] = 2 * layers
    out["workload"] = (f"{layers} layers x svd_kv_attention: {Hq} query heads, {Hkv} kv heads, "
                       f"dim {D}, K+1 = {C}, keys q8_0 / values q4_0, one cache per layer")
    return out


def lm_head_windows(vp, dev, peak, n_windows=10000, C=6, pool=16, seed=23):
    """The lm_head + sampler workload with sampled acceptance: n_windows verify windows of K+1 = C
    positions, each the 5120 x 151936 lm_head over the window's C hidden columns with the
    production sampler (svd_lm_head_softmax) and then svd_accept of the window's C - 1 drafts
    against a drafter q drawn from the target's perturbed logits (stack.DRAFTER_SIGMA, alpha about
    0.5).  The hidden columns come from a pool of `pool` synthetic windows, the drafter's rows and
    drafts are made from each pool entry once (untimed), and the timed loop runs the windows back
    to back on the resident lm_head.  Reports windows/s, the lm_head's weight stream per window
    against the copy peak and the tokens emitted per window."""
    import torch

    from speculative_decoding_verify_06_gb300 import stack, svd, synth
    V, k, hid = synth.VOCAB, C - 1, synth.HIDDEN
    W = vp.lm.W
    smp = vp.sampler
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    Hs = [synth.activations_torch(C, hid, seed * 1000 + i, dev) for i in range(pool)]
    logits = torch.empty((C, V), dtype=torch.float32, device=dev)
    probs = torch.empty_like(logits)
    am = torch.empty(C, dtype=torch.int32, device=dev)
    ws = torch.zeros(svd.svd_lm_head_workspace_bytes(hid, V, C), dtype=torch.uint8, device=dev)
    qws = torch.zeros(svd.svd_sampler_workspace_bytes(k, V), dtype=torch.uint8, device=dev)
    qam = torch.empty(k, dtype=torch.int32, device=dev)
    qs, drafts = [], []
    for H in Hs:  # the drafter of each pool window (untimed)
        svd.svd_lm_head_softmax(W, H, C, smp, logits, probs, am, ws)
        noise = torch.empty((k, V), dtype=torch.float32, device=dev)
        noise.normal_(0.0, stack.DRAFTER_SIGMA, generator=g)
        q = torch.empty((k, V), dtype=torch.float32, device=dev)
        svd.svd_sampler_probs((logits[:k] + noise).contiguous(), k, V, smp, q, qam, qws)
        qs.append(q)
        drafts.append(torch.multinomial(q, 1, generator=g).to(torch.int32).view(1, k).contiguous())
    tok = torch.empty((n_windows, k + 1), dtype=torch.int32, device=dev)
    ne = torch.empty(n_windows, dtype=torch.int32, device=dev)
    st = torch.empty(n_windows, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream(dev)

    def window(w):
        i = w % pool
        svd.svd_lm_head_softmax(W, Hs[i], C, smp, logits, probs, am, ws, stream=s)
        svd.svd_accept(probs, drafts[i], 1, k, V, tok[w], ne[w:w + 1], st[w:w + 1], q=qs[i],
                       seed=seed, window_offset=w, stream=s)
    for w in range(3):
        window(w)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for w in range(n_windows):
        window(w)
    e1.record(s)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    per = ms / n_windows
    wbytes = roofline_lm_bytes(hid, V, C)
    out = {"windows": n_windows, "C": C, "ms_per_window": per, "windows_per_s": 1000.0 / per,
           "lm_head_gb_s": wbytes / per / 1e6, "frac": wbytes / per / 1e6 / peak,
           "tokens_per_window": float(ne.double().mean().item()),
           "status_nonzero": int((st != 0).sum().item()),
           "launches_per_window": 3,
           "workload": (f"{n_windows} windows: lm_head {hid} x {V} over K+1 = {C} columns + sampler "
                        f"(T 0.6, top-p 0.95, min-p 0.05) over {C} rows + svd_accept of {k} drafts "
                        f"against the drafter's q (target logits + N(0, sigma^2), alpha about 0.5); "
                        f"{pool} synthetic windows cycled")}
    del Hs, qs, drafts, logits, probs, ws
    torch.cuda.empty_cache()
    return out


def roofline_lm_bytes(hid, V, C):
    """Algorithmic bytes of one lm_head window: the weights and scales once, the C hidden columns
    in and the C logit rows out."""
    from speculative_decoding_verify_06_gb300 import roofline
    return roofline.linear_bytes(hid, V, C)


def q4k_stack(dev, peak, tail_ms, layers=64, C=4, steps=20, oracle_sample=False):
    """The stack with Q4_K super-block weights (stack.Q4kStack: the pages' checkpoint format,
    repacked once into the Q4_K native layout; one chain launch in a CUDA graph), timed like the
    main stack; the pass rate adds the lm_head/sampler/acceptance tail of the main timed region."""
    import torch

    from speculative_decoding_verify_06_gb300 import stack, svd
    qs = stack.Q4kStack(layers=layers, C=C, seed=11, device=dev).capture()
    s = torch.cuda.current_stream(dev)
    for _ in range(3):
        qs.launch(s)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        qs.launch(s)
    e1.record(s)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    nbytes = qs.stack_bytes()
    rc, bits = svd.svd_verify_status(qs.ws)
    traffic = kernel_traffic("vl_stream_kernel_q4k_27b_stack_c4.txt") if (layers == 64 and C == 4) else None
    out = {"C": C, "stack_ms": ms, "bytes": nbytes, "gb_s": nbytes / ms / 1e6,
           "frac": nbytes / ms / 1e6 / peak, "passes_per_s": 1000.0 / (ms + tail_ms),
           "traffic": traffic,
           "status_bits": bits,
           "kernel": "vl_stream_kernel on Q4_K units (64 rows x 256 inputs), one chain launch",
           "workload": (f"{layers} layers x (q|k|v 5120->7168, o 5120->5120, gate|up "
                        "5120->34816, down 17408->5120) in Q4_K super-blocks (fp16 d, dmin, "
                        "6-bit sub-block scales and mins, 4-bit codes), C = K+1 = 4")}
    del qs
    torch.cuda.empty_cache()
    if oracle_sample:
        out["cpu_baseline"] = q4k_oracle_sample()
    return out


def q4k_oracle_sample(out_f=5120, in_f=5120, C=4, seed=12):
    """The Q4_K oracle (fp64 numpy: dequantisation of every weight, then the product) on one
    o-projection-shaped matrix, as Q4_K bytes per second."""
    from oracle import kquant
    from speculative_decoding_verify_06_gb300 import synth
    blocks = synth.q4k_blocks(out_f, in_f, seed)
    x = synth.activations(C, in_f, seed + 1)
    t0 = time.perf_counter()
    kquant.verify_linear(blocks, in_f, x)
    dt = time.perf_counter() - t0
    nbytes = out_f * (in_f // 256) * 144 + C * in_f * 2 + C * out_f * 4
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "seconds": dt,
            "sample": (f"one {in_f}->{out_f} Q4_K matrix at C = {C} through oracle/kquant.py "
                       "(fp64 numpy; the product on the BLAS threads numpy was built with, up to "
                       "the host's cores); GB/s of its algorithmic bytes")}


def pass_with_kv(vp, dev, peak, tail_ms, context=32768, steps=20):
    """The verify pass with each layer's KV cache in its place (stack.KvPass: the window's keys
    and values appended, then attention over the layer's own cache, between its q|k|v and o
    products; the matrices between two attention steps in one chain launch; one CUDA graph), at
    the pages' 32K context, plus the lm_head/sampler/acceptance tail measured in the main timed
    region.  Reports the pass rate and the bytes of weights and cache per second."""
    import torch

    from speculative_decoding_verify_06_gb300 import stack
    kp = stack.KvPass(vp, context).capture()
    s = torch.cuda.current_stream(dev)
    for _ in range(3):
        kp.launch(s)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        kp.launch(s)
    e1.record(s)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    nbytes = vp.stack_bytes() + kp.kv_bytes()
    out = {"context": context, "stack_with_kv_ms": ms, "tail_ms": tail_ms,
           "passes_per_s": 1000.0 / (ms + tail_ms), "bytes": nbytes,
           "gb_s": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / peak,
           "launches_per_pass": kp.launches(),
           "workload": ("per layer, between its q|k|v and o products: svd_kv_attention_append "
                        "(the window's keys and values from the q|k|v output quantised into the "
                        "layer's own q8_0-key / q4_0-value cache, then 40 query heads over 8 kv "
                        "heads of dim 128 attending over it, one kernel); the matrices between "
                        "two attention steps in one chain launch (65 chain launches per pass); "
                        "one CUDA graph")}
    del kp
    torch.cuda.empty_cache()
    return out


def run_svd(args, rank, world, local_rank):
    import torch

    from speculative_decoding_verify_06_gb300 import build, roofline, stack, svd, synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    build.build_library()
    vp = stack.VerifyPass(layers=args.layers, C=args.C, seed=rank, device=dev, pdl=not args.no_pdl,
                          chain=not args.no_chain, head=not args.stack_only)
    vp.capture()
    s = torch.cuda.current_stream(dev)
    dist = world > 1
    if dist:
        import torch.distributed as td

    for _ in range(args.warmup):
        vp.launch(s)
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if dist:
        td.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(_gpu_id(dev)) as clk:
        for i in range(K):
            ev[i][0].record(s)
            vp.launch(s, ev_mid=ev[i][1])
            ev[i][2].record(s)
        torch.cuda.synchronize(dev)
    if dist:
        td.barrier()
    total_ms = ev[0][0].elapsed_time(ev[-1][2])
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    stack_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    tail_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    t_max = max_over_ranks(total_ms, dev)
    passes_per_s = replica_rate(K, world, t_max)

    # tokens per pass of this window's (p, q): 20k windows drawn from the same rows (untimed)
    tokens_per_pass = None
    if vp.accept:
        n_win = 20000
        k, V = vp.k, vp.V
        gen = torch.Generator(device=dev)
        gen.manual_seed(4242 + rank)
        drafts = torch.multinomial(vp.q, n_win, replacement=True, generator=gen).T.contiguous().to(torch.int32)
        p_rows = torch.arange(k + 1, device=dev, dtype=torch.int64).repeat(n_win, 1)
        q_rows = torch.arange(k, device=dev, dtype=torch.int64).repeat(n_win, 1)
        tok = torch.empty((n_win, k + 1), dtype=torch.int32, device=dev)
        ne = torch.empty(n_win, dtype=torch.int32, device=dev)
        st = torch.empty(n_win, dtype=torch.int32, device=dev)
        svd.svd_accept(vp.probs, drafts, n_win, k, V, tok, ne, st, q=vp.q, p_rows=p_rows,
                       q_rows=q_rows, seed=rank + 17)
        torch.cuda.synchronize(dev)
        tokens_per_pass = float(ne.double().mean().item())

    # end to end: inputs from pinned host memory and the result back, every step
    host_in = [t.detach().cpu().pin_memory() for t in vp.inputs()]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in vp.outputs()]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    Ke = max(1, min(K, args.e2e_steps))
    if dist:
        td.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(s)
    for _ in range(Ke):
        for d_t, h_t in zip(vp.inputs(), host_in):
            d_t.copy_(h_t, non_blocking=True)
        vp.launch(s)
        for h_t, d_t in zip(host_out, vp.outputs()):
            h_t.copy_(d_t, non_blocking=True)
    e1.record(s)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - w0
    e2e_ms = max_over_ranks(max(e0.elapsed_time(e1), wall * 1000.0), dev)
    e2e_value = replica_rate(Ke, world, e2e_ms)

    stack_bytes = vp.stack_bytes()
    achieved = stack_bytes / (stack_ms / 1000.0) / 1e9
    peak, peak_kind = peaks()
    traffic_pass = kernel_traffic()
    n_launch = len(vp.linears)
    line = {
        "metric": METRIC, "value": passes_per_s, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "C": args.C, "layers": args.layers,
                   "global_batch": world, "parallelism": f"replicas{world}",
                   "l2": (f"inputs larger than L2: {vp.stack_bytes() / 1e9:.1f} GB of weights "
                          f"streamed per step"),
                   "stack_launch": ("per-matrix launches, PDL" if args.no_chain else
                                    f"one persistent cooperative chain of {len(vp.linears)} "
                                    f"matrices"),
                   "graph": "stack graph + tail graph per step",
                   "stack_only": bool(args.stack_only)},
        "stack": {"ms": stack_ms, "passes_per_s": 1000.0 / stack_ms, "bytes": stack_bytes,
                  "gb_s": achieved, "tail_ms": tail_ms},
        "step_ms": percentiles(step_ms),
        "tokens_per_pass": tokens_per_pass,
        "effective_tokens_per_s": (None if tokens_per_pass is None else
                                   passes_per_s * tokens_per_pass),
        "pass_bytes": vp.pass_bytes(),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "kernel": "vl_stream_kernel (one chain launch: the stack's 256 matrices)",
                     "traffic": None if traffic_pass is None else traffic_pass},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke,
                "copies": ("per step, from pinned host memory: the first layer's input (the "
                           "embedded window), the drafter's q rows and the drafts; back: the "
                           "emitted tokens, their count and the status word")},
        # per step: the stack (one chain launch, or one per matrix), the lm_head, the sampler
        # (one cluster launch) and the acceptance
        "gpu_launches": K * ((n_launch if args.no_chain else 1) + (1 + 1 + 1 if vp.head else 0)),
        "clocks": clk.summary(),
    }
    if not args.no_sweep and not args.stack_only:
        line["column_sweep"] = column_sweep(vp, dev, 20, tokens_per_pass, peak)
        line["accept_throughput"] = accept_throughput(
            dev, peak, oracle_windows=2000 if (rank == 0 and world == 1
                                               and not args.no_cpu_baseline) else 0)
    if not args.no_sweep and not args.stack_only and vp.head:
        line["lm_head_windows"] = lm_head_windows(vp, dev, peak)
    if not args.no_kv and not args.stack_only:
        line["kv_read"] = kv_read(dev, peak, line["stack"]["ms"], layers=args.layers,
                                  contexts=tuple(int(c) for c in args.kv_contexts.split(",")),
                                  oracle_sample=(rank == 0 and world == 1
                                                 and not args.no_cpu_baseline))
        line["pass_with_kv"] = pass_with_kv(vp, dev, peak, line["stack"]["tail_ms"])
    if not args.no_q4k and not args.stack_only:
        line["q4k_stack"] = q4k_stack(dev, peak, line["stack"]["tail_ms"], layers=args.layers,
                                      C=args.C if args.C <= 8 else 4,
                                      oracle_sample=(rank == 0 and world == 1
                                                     and not args.no_cpu_baseline))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample()  # one whole pass on every host thread
        times = [smp.step()]
        one = OracleSample(layers=1, threads=1)  # a bounded single-thread sample
        t1 = [one.step()]
        line["cpu_baseline"] = {"value": smp.passes_per_s(times), "unit": UNIT,
                                "cores": smp.threads, "kind": "oracle", "sample": smp.describe(1),
                                "seconds": times[0], "cpu": _cpu_model(),
                                "single_thread": {"value": one.passes_per_s(t1), "cores": 1,
                                                  "sample": one.describe(1), "seconds": t1[0]}}
        if not args.stack_only:
            line["lm_head_window_cpu_baseline"] = lm_head_oracle_windows()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="svd", choices=["svd", "reference"])
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--C", type=int, default=4)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-chain", action="store_true",
                    help="one launch per matrix (with PDL) instead of the persistent chain")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kv", action="store_true",
                    help="skip the KV-read measurement (attention over q8_0/q4_0 caches)")
    ap.add_argument("--kv-only", action="store_true",
                    help="print only the KV-read measurement")
    ap.add_argument("--kv-contexts", default=",".join(str(c) for c in KV_CONTEXTS),
                    help="comma-separated context lengths of the KV-read measurement")
    ap.add_argument("--no-q4k", action="store_true",
                    help="skip the stack in Q4_K super-block weights")
    ap.add_argument("--q4k-only", action="store_true",
                    help="print only the Q4_K stack measurement (for profiling small stacks)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the window-width sweep and the acceptance-throughput sample")
    ap.add_argument("--stack-only", action="store_true",
                    help="time the layer stack alone (no lm_head, sampler or acceptance); for "
                         "profiling small stacks")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.kv_only:
        import torch

        from speculative_decoding_verify_06_gb300 import build
        build.build_library()
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        peak, _ = peaks()
        ctxs = tuple(int(c) for c in args.kv_contexts.split(","))
        print(json.dumps({"kv_read": kv_read(dev, peak, None, layers=args.layers,
                                             contexts=ctxs, steps=args.steps)}), flush=True)
        return
    if args.q4k_only:
        import torch

        from speculative_decoding_verify_06_gb300 import build
        build.build_library()
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        peak, _ = peaks()
        print(json.dumps({"q4k_stack": q4k_stack(dev, peak, 0.0, layers=args.layers,
                                                 C=args.C, steps=args.steps)}), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as td
        torch.cuda.set_device(local_rank)
        td.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    run_svd(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as td
        td.destroy_process_group()


if __name__ == "__main__":
    main()
