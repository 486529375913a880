"""Benchmark: ERI quartets/s and FP64 GFLOP/s per angular class on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload homogeneous|high_l|g_shells|deriv|classes|cluster64|cluster200|cluster64_jk|
                                cluster200_jk|cluster64_store|ladder_f_jk|deriv_f]
                    [--scale S] [--ablation all|NAME,...]

A step is one pass of the hot path over the workload's batch: for every class
of the workload, the class kernel evaluates all its quartets (Gaussian-pair
parameters, Boys function, VRR, contraction, HRR with the stepwise spherical
transform, block store).  ``value`` is the whole job's shell quartets per second
with inputs resident in HBM; ``e2e`` is the same metric through the C ABI with
host buffers (every step: plan creation from host shells, pinned host->device
copy of the quartet lists, device->host copy of every block into pinned host
memory; the class batches on separate streams so that their host and device
work overlap).  ``--ablation`` builds and times the generator-ablation
libraries (electron_repulsion_integrals_gb300/ablation.py) against the main one.

Default workload (N=1): the homogeneous class batch, 1,048,576 (pp|pp) and
1,048,576 (dd|dd) quartets, centers uniform in a 10 bohr cube, exponents
log-uniform in [0.05, 100], contraction degree 1, spherical output.

Under torchrun each rank runs the same per-GPU batch on its own GPU (replicas:
quartets are independent, there is no data-path collective); ``value`` is the
total quartets of all ranks over the slowest rank's time ("scaling": "weak").

``--impl reference`` times the CPU oracle (oracle/, McMurchie-Davidson in
C++/OpenMP) on the host cores on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ERI quartets/s and FP64 GFLOP/s per angular class (fraction of GB300 FP64 peak)"
# FP64 pipe rate from unit counts and clock (152 SMs x 2 DFMA/clk x 2 flop x
# 2.070 GHz): used only when the measured probe is unavailable
FP64_PEAK_NOMINAL_TFLOPS = 152 * 2 * 2 * 2.070e9 / 1e12
E2E_CHUNK_BYTES = 0.75e9  # output bytes per e2e chunk: readback of one overlaps compute of the next
E2E_TAIL_BYTES = 0.1e9    # output bytes of the last e2e chunk, whose readback nothing overlaps

WORKLOADS = {
    "homogeneous": {"desc": "homogeneous class batch: (pp|pp) x 1,048,576 + (dd|dd) x 1,048,576 quartets, "
                            "centers U[0,10]^3 bohr, exponents log-U[0.05,100], degree 1, spherical",
                    "classes": [((1, 1, 1, 1), 1 << 20, 1, 1), ((2, 2, 2, 2), 1 << 20, 1, 101)]},
    "high_l": {"desc": "high-L batch: (ff|ff) x 131,072 + (fd|fd) x 262,144 quartets, degree 2, spherical",
               "classes": [((3, 3, 3, 3), 131072, 2, 2), ((3, 2, 3, 2), 262144, 2, 102)]},
    "g_shells": {"desc": "g-shell batch: (gg|gg) x 16,384 + (gd|gd) x 65,536 quartets, degree 2, centers U[0,10]^3 "
                         "bohr, exponents log-U[0.05,100], spherical",
                 "classes": [((4, 4, 4, 4), 16384, 2, 3), ((4, 2, 4, 2), 65536, 2, 103)]},
    "deriv": {"desc": "first derivatives (12 blocks per quartet): (pp|pp) x 524,288 + (dd|dd) x 131,072 quartets, "
                      "degree 1, centers U[0,10]^3 bohr, exponents log-U[0.05,100], spherical",
              "classes": [((1, 1, 1, 1), 1 << 19, 1, 4), ((2, 2, 2, 2), 1 << 17, 1, 104)], "deriv": True},
    "deriv_f": {"desc": "first derivatives of f-shell classes (12 blocks per quartet): (fd|fd) x 16,384 + (ff|ff) x "
                        "4,096 quartets, degree 1, centers U[0,10]^3 bohr, exponents log-U[0.05,100], spherical",
                "classes": [((3, 2, 3, 2), 1 << 14, 1, 105), ((3, 3, 3, 3), 1 << 12, 1, 106)], "deriv": True},
    "classes": {"desc": "every canonical class of s, p, d, f shells through (ff|ff) (55 classes), contraction "
                        "degree 1 and 2, centers U[0,10]^3 bohr, exponents log-U[0.05,100], spherical; quartets per "
                        "class sized to about 8 GFLOP per launch"},
    "cluster64": {"desc": "64-atom synthetic cluster (radius 12 bohr, 32 heavy 3s2p1d + 32 light 2s1p, 1-6 "
                          "primitives, exponents log-U[0.1,5000]): Coulomb J over all unique quartets surviving "
                          "Schwarz 1e-10, spherical, D = C C^T", "cluster": (64, 3)},
    "cluster200": {"desc": "200-atom synthetic cluster (same composition), Coulomb J over all unique quartets "
                           "surviving Schwarz 1e-10, spherical, D = C C^T (C: N x N/4, N(0,1)/sqrt(N))",
                   "cluster": (200, 4)},
    "cluster64_jk": {"desc": "64-atom synthetic cluster as cluster64: Coulomb J and exchange K together in one "
                             "pass over all unique quartets surviving Schwarz 1e-10", "cluster": (64, 3), "jk": True},
    "cluster200_jk": {"desc": "200-atom synthetic cluster as cluster200: Coulomb J and exchange K together in one "
                              "pass over all unique quartets surviving Schwarz 1e-10", "cluster": (200, 4),
                      "jk": True},
    "ladder_f_jk": {"desc": "16-atom synthetic cluster (radius 6 bohr, atoms >= 2 bohr apart) with one s, p, d and f "
                            "shell per atom (1-3 primitives, exponents log-U[0.1,50]): Coulomb J and exchange K in one "
                            "pass over all unique quartets surviving Schwarz 1e-10, spherical, D = C C^T; the "
                            "cooperative tier's digestion", "cluster": (16, 842), "ladder": (3, 6.0, 2.0), "jk": True},
    "cluster64_store": {"desc": "64-atom synthetic cluster as cluster64: every unique quartet surviving Schwarz 1e-10 "
                                "computed and stored, spherical, one eri_compute_screened launch per class",
                        "cluster": (64, 3), "store": True},
}


def dram_traffic(cls, n, deriv=False):
    """DRAM bytes of one launch of the class kernel (the derivative kernel with
    deriv) from its ncu record in profiles/dram_traffic.json (captured on a
    slice and scaled by the number of quartets, the traffic being per quartet),
    or None without a record or when the kernel sources changed since the
    capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    name = "k_{}{}{}{}{}".format("d" if deriv else "c", *cls)
    recs = [r for r in json.load(open(path)) if r["kernel"].split()[0] == name]
    if not recs:
        return None
    rec = recs[0]
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, "electron_repulsion_integrals_gb300", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != rec["sha256"]:
        return None
    return rec["dram_bytes_per_quartet"] * n


def e2e_chunks(n, out_bytes):
    """Quartet ranges [lo, hi) covering 0..n in order: about E2E_CHUNK_BYTES of
    output each (at most 8), and, when the batch is larger than
    4 E2E_TAIL_BYTES, a last range of about E2E_TAIL_BYTES: a chunk's readback
    overlaps the next chunk's compute, so only the last readback is exposed
    (device-to-host runs at about 193 GB/s here, a 0.75 GB chunk at 3.9 ms)."""
    tail = 0
    if out_bytes > 4 * E2E_TAIL_BYTES and n >= 2:
        tail = max(1, min(n - 1, int(E2E_TAIL_BYTES * n / out_bytes)))
    m = n - tail
    k = max(1, min(8 - (1 if tail else 0), m, round((out_bytes * m / n) / E2E_CHUNK_BYTES)))
    out = [(m * j // k, m * (j + 1) // k) for j in range(k)]
    if tail:
        out.append((m, n))
    return out


def max_over_ranks(ms, dist, device):
    """The slowest rank's time (all ranks receive it); ms itself without a
    process group."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rate(per_rank_units, world, steps, ms):
    """Whole-job throughput of replicas: every rank processes per_rank_units
    per step; the job takes the slowest rank's time."""
    return per_rank_units * world * steps / (ms / 1e3)


def env_int(k, d):
    try:
        return int(os.environ.get(k, d))
    except ValueError:
        return d


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measure_fp64_peak(dev, stream, gpu_index, target_s=0.4):
    """FP64 pipe rate on this GPU: eri_fp64_probe (independent FMA chains,
    8 blocks of 256 threads per SM) timed with CUDA events on `stream`, SM clock
    sampled meanwhile.  Returns TFLOP/s (2 flops per FMA) and the median clock."""
    import torch
    import electron_repulsion_integrals_gb300 as eri
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, threads = nsm * 8, 256
    sink = torch.empty(blocks * threads, dtype=torch.float64, device=dev)

    def timed(iters, reps=1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fmas = 0
        for _ in range(reps):
            fmas += eri.eri_fp64_probe("fma", blocks, threads, iters, sink, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        return fmas, e0.elapsed_time(e1)

    timed(2000)
    fmas, ms = timed(2000)
    iters = int(min(4e6, max(2000, 2000 * (target_s / 4) / max(ms / 1e3, 1e-6))))
    clocks = ClockSampler(gpu_index)
    clocks.start()
    time.sleep(0.3)
    fmas, ms = timed(iters, 4)
    clk = clocks.stop()
    return {"tflops": 2 * fmas / (ms / 1e3) / 1e12, "sm_mhz": clk.get("sm_mhz"), "reasons": clk.get("reasons"),
            "ms": ms, "fmas": fmas, "grid": f"{blocks} x {threads} threads, 8 FMA chains each"}


def run_fp64_peak(a, local_rank):
    """The FP64 probe over launch shapes (threads per block x blocks per SM,
    8 independent chains per thread) and, at one shape, FMA vs MUL vs ADD:
    one JSON line with the rates (G operations/s) and the SM clock."""
    import torch
    import electron_repulsion_integrals_gb300 as eri
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    eri.lib()
    stream = torch.cuda.current_stream()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.empty(nsm * 2048, dtype=torch.float64, device=dev)

    def rate(op, threads, bps, target_ops=1.5e11):
        blocks = nsm * bps
        iters = int(target_ops / (blocks * threads * 8))
        eri.eri_fp64_probe(op, blocks, threads, 100, sink, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = eri.eri_fp64_probe(op, blocks, threads, iters, sink, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        return n / (e0.elapsed_time(e1) / 1e3) / 1e9

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    shapes = {}
    for threads in (64, 128, 256, 512):
        for bps in (1, 2, 4, 8):
            if threads * bps <= 2048:
                shapes[f"{threads}x{bps}"] = rate("fma", threads, bps)
    ops = {op: rate(op, 256, 4) for op in ("fma", "mul", "add")}
    clk = clocks.stop()
    best = max(shapes.values())
    print(json.dumps({"metric": "FP64 pipe rate (eri_fp64_probe)", "unit": "G operations/s", "nsm": nsm,
                      "fma_by_shape_threads_x_blocks_per_sm": shapes, "by_op_256x4": ops,
                      "peak_tflops": 2 * best / 1e3, "clocks": clk}), flush=True)


def roofline_peak(probe, timed_mhz):
    """The FP64 peak for a timed region: the probe's measured rate scaled from
    its median SM clock to the region's, or the nominal figure without a probe."""
    if not probe or not probe.get("tflops"):
        return FP64_PEAK_NOMINAL_TFLOPS, "nominal FP64 pipe: 152 SMs x 2 DFMA/clk x 2 flop x 2.07 GHz"
    p = probe["tflops"]
    src = f"measured: eri_fp64_probe (FMA chains) {p:.4g} TFLOP/s"
    if probe.get("sm_mhz") and timed_mhz:
        p *= timed_mhz / probe["sm_mhz"]
        src += f" at {probe['sm_mhz']:.0f} MHz, scaled to the timed region's {timed_mhz:.0f} MHz"
    return p, src


def cpu_oracle_rate(wl, budget_s=20.0, nthreads=None):
    """Oracle time per quartet for each class of the workload from a bounded
    sample; returns (quartets/s for the whole step mix, description, cores)."""
    import oracle
    from electron_repulsion_integrals_gb300 import workloads as W
    nthreads = nthreads or oracle.default_threads()
    per_class = {}
    total_time = 0.0
    total_q = 0
    parts = []
    share = budget_s / len(wl["classes"])
    for cls, n, deg, seed in wl["classes"]:
        m = 64
        spent = 0.0
        done = 0
        while spent < share:
            s, q = W.homogeneous(cls, m, deg, seed_index=seed + 7000 + done)
            S = oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)
            t0 = time.perf_counter()
            if wl.get("deriv"):
                oracle.eri_deriv_blocks(S, q, spherical=True, nthreads=nthreads)
            else:
                oracle.eri_blocks(S, q, spherical=True, nthreads=nthreads)
            dt = time.perf_counter() - t0
            spent += dt
            done += m
            if dt < share / 8:
                m *= 2
        tq = spent / done
        per_class[cls] = tq
        total_time += tq * n
        total_q += n
        parts.append(f"{done} {cls} quartets")
    return total_q / total_time, "oracle on " + " + ".join(parts), nthreads, per_class


def oracle_cluster_counts(s, tau=1e-10):
    """Unique shell quartets per canonical class that pass Q_ab Q_cd >= tau
    with the oracle's Schwarz factors (counted from the sorted pair factors,
    not listed)."""
    import oracle
    Q = oracle.schwarz(oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs), spherical=True)
    L = np.asarray(s.L)
    a, b = np.tril_indices(s.n)
    hi, lo = np.maximum(L[a], L[b]), np.minimum(L[a], L[b])
    pc = hi * (hi + 1) // 2 + lo
    groups = {int(k): (int(hi[pc == k][0]), int(lo[pc == k][0]), np.sort(Q[a, b][pc == k])) for k in np.unique(pc)}
    counts = {}
    with np.errstate(divide="ignore"):
        for cb, (la, lb, qb) in groups.items():
            for ck, (lc, ld, qk) in groups.items():
                if ck > cb:
                    continue
                ge = len(qk) - np.searchsorted(qk, tau / qb, side="left")  # ket factors >= tau / Q_bra
                n = int(ge.sum())
                if ck == cb:
                    n = (n + int(np.count_nonzero(qb * qb >= tau))) // 2
                counts[(la, lb, lc, ld)] = n
    return counts


def run_reference(a, rank, world):
    wl = WORKLOADS[a.workload]
    if rank != 0:
        return
    rates = []
    desc = ""
    cores = 0
    if "cluster" in wl:
        cs = cluster_shells(wl)
        counts = oracle_cluster_counts(cs)
        rate_fn = lambda budget: cpu_oracle_rate_cluster(cs, counts, budget_s=budget) + (None,)  # noqa: E731
    else:
        rate_fn = lambda budget: cpu_oracle_rate(wl, budget_s=budget)  # noqa: E731
    # each step a bounded sample: about two minutes for the whole timed run
    budget = max(2.0, min(a.ref_budget, 120.0 / max(a.steps, 1)))
    for _ in range(a.warmup):
        rate_fn(2.0)
    t_all = time.perf_counter()
    for _ in range(a.steps):
        r, desc, cores, _ = rate_fn(budget)
        rates.append(r)
    elapsed = time.perf_counter() - t_all
    value = statistics.median(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "quartets/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": elapsed / a.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl["desc"]},
            "cpu_baseline": {"value": value, "unit": "quartets/s", "cores": cores, "kind": "oracle",
                             "sample": desc + " per step, projected to the full step mix"},
            "e2e": {"value": value, "unit": "quartets/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cluster_shells(wl):
    """Shells of a cluster workload."""
    from electron_repulsion_integrals_gb300 import workloads as W
    natom, idx = wl["cluster"]
    if "ladder" in wl:
        lmax, radius, dmin = wl["ladder"]
        return W.shell_ladder_cluster(natom, lmax, seed_index=idx, radius=radius, dmin=dmin)
    return W.cluster(natom, seed_index=idx)


def run_coulomb(a, rank, world, local_rank):
    """Cluster workloads: one step = eri_build_J (or eri_build_JK) over every surviving unique quartet."""
    import torch
    import electron_repulsion_integrals_gb300 as eri
    from electron_repulsion_integrals_gb300 import workloads as W
    from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    eri.lib()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[a.workload]
    idx = wl["cluster"][1]
    s = cluster_shells(wl)
    nbf = W.nbf(s)
    D = W.density(nbf, idx)
    stream = torch.cuda.current_stream()
    t = time.perf_counter()
    plan = eri.Plan(s, spherical=True, schwarz_tau=1e-10, stream=stream)
    plan_s = time.perf_counter() - t
    counts = {c: plan.quartet_count(c) for c in canonical_classes(int(s.L.max()))}
    nq = sum(counts.values())
    Dd = torch.as_tensor(D, device=dev)
    J = torch.empty_like(Dd)
    K = torch.empty_like(Dd)
    jk = bool(wl.get("jk"))

    def digest():
        if jk:
            plan.build_JK(Dd, J, K, stream)
        else:
            plan.build_J(Dd, J, stream)

    probe = measure_fp64_peak(dev, stream, local_rank)
    for _ in range(a.warmup):
        digest()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(a.steps):
        digest()
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    ms = max_over_ranks(ms, dist, dev)
    value = replica_rate(nq, world, a.steps, ms)
    # algorithmic flops: per class, quartets x (primitive quartets x VRR + HRR) + per digested integral
    # 2 FMA for J (+ 4 FMA for K)
    prim_q = 0.0
    flops = 0.0
    per_class = {}
    for c, n in counts.items():
        if n == 0:
            continue
        st = eri.eri_class_info(c)
        _, pq = eri.eri_plan_class_work(plan.handle, c)
        prim_q += pq
        flops += pq * st["vrr_flops"] + n * (st["hrr_flops"] + (12 if jk else 4) * eri.block_size(c))
        per_class["({}{}|{}{})".format(*c)] = {"quartets": n, "primitive_quartets": pq}
    ach = flops / (ms / a.steps / 1e3) / 1e12
    peak, peak_src = roofline_peak(probe, clk.get("sm_mhz"))
    e2e = None
    if a.e2e:
        hD = torch.from_numpy(D).pin_memory()
        hJ = torch.empty(hD.shape, dtype=torch.float64, pin_memory=True)
        hK = torch.empty(hD.shape, dtype=torch.float64, pin_memory=True)
        torch.cuda.synchronize()
        te = time.perf_counter()
        p2 = eri.Plan(s, spherical=True, schwarz_tau=1e-10, stream=stream)
        dd = hD.to(dev, non_blocking=True)
        if jk:
            Jd, Kd = p2.build_JK(dd, None, None, stream)
            hK.copy_(Kd, non_blocking=True)
        else:
            Jd = p2.build_J(dd, None, stream)
        hJ.copy_(Jd, non_blocking=True)
        torch.cuda.synchronize()
        te = time.perf_counter() - te
        p2.close()
        e2e = {"value": nq * world / te, "unit": "quartets/s", "h2d_bytes_per_step": hD.numel() * 8 + s.n * 48 +
               s.exps.size * 16, "d2h_bytes_per_step": hJ.numel() * 8 * (2 if jk else 1)}
    cpu = None
    if rank == 0 and a.cpu_baseline:
        rate, desc, cores = cpu_oracle_rate_cluster(s, counts, budget_s=a.ref_budget)
        cpu = {"value": rate, "unit": "quartets/s", "cores": cores, "kind": "oracle", "sample": desc}
    line = {"metric": METRIC, "value": value, "unit": "quartets/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "per_class": per_class,
            "config": {"workload": wl["desc"], "unique_quartets": nq, "primitive_quartets": prim_q, "nbf": nbf,
                       "plan_create_s": plan_s, "l2": "no flush: J digestion re-reads D; kernels are FP64-bound",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "alu", "kernel": "all class kernels of " + ("eri_build_JK" if jk else "eri_build_J"), "achieved": ach,
                         "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                         "traffic": None, "peak_source": peak_src},
            "fp64_probe": probe, "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": a.steps * (sum(1 for n in counts.values() if n) + (2 if jk else 1))}
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if dist:
        dist.destroy_process_group()


def run_store(a, rank, world, local_rank):
    """Cluster store workload: one step = eri_compute_screened over every
    class's screened unique quartets, blocks stored into per-class device
    buffers (eri_plan_class_quartets gives the shells of each block)."""
    import torch
    import electron_repulsion_integrals_gb300 as eri
    from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    eri.lib()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[a.workload]
    s = cluster_shells(wl)
    stream = torch.cuda.current_stream()
    t = time.perf_counter()
    plan = eri.Plan(s, spherical=True, schwarz_tau=1e-10, stream=stream)
    plan_s = time.perf_counter() - t
    counts = {c: plan.quartet_count(c) for c in canonical_classes(int(s.L.max()))}
    classes = [c for c, n in counts.items() if n]
    outs = {}
    prim_q = {}
    for c in classes:
        outs[c] = torch.empty(counts[c] * eri.block_size(c), dtype=torch.float64, device=dev)
        prim_q[c] = eri.eri_plan_class_work(plan.handle, c)[1]
    nq = sum(counts[c] for c in classes)
    out_bytes = sum(o.numel() * 8 for o in outs.values())
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(classes) + 1)]

    def step(record=False):
        if record:
            ev[0].record(stream)
        for i, c in enumerate(classes):
            eri.eri_compute_screened(plan.handle, c, 0, counts[c], outs[c], stream)
            if record:
                ev[i + 1].record(stream)

    probe = measure_fp64_peak(dev, stream, local_rank)
    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(a.steps):
        step(record=(k == a.steps - 1))
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    ms = max_over_ranks(ms, dist, dev)
    value = replica_rate(nq, world, a.steps, ms)
    flops = 0.0
    per_class = {}
    for i, c in enumerate(classes):
        st = eri.eri_class_info(c)
        f = prim_q[c] * st["vrr_flops"] + counts[c] * st["hrr_flops"]
        flops += f
        cms = ev[i].elapsed_time(ev[i + 1])
        per_class["({}{}|{}{})".format(*c)] = {"quartets": counts[c], "primitive_quartets": prim_q[c],
                                               "ms_per_launch": cms, "quartets_per_s": counts[c] / (cms / 1e3),
                                               "fp64_gflops": f / (cms / 1e3) / 1e9,
                                               "tier": "staged" if st["staged"] else "register"}
    ach = flops / (ms / a.steps / 1e3) / 1e12
    peak, peak_src = roofline_peak(probe, clk.get("sm_mhz"))
    e2e = None
    if a.e2e:
        # public API end to end: plan from host shells, every class's blocks
        # and its quartet list (the shells of each block) computed and read
        # back into pinned host memory (each class's readback on a copy
        # stream overlaps the next class's compute)
        host = {c: torch.empty(o.numel(), dtype=torch.float64, pin_memory=True) for c, o in outs.items()}
        hlist = {c: torch.empty((counts[c], 4), dtype=torch.int32, pin_memory=True) for c in classes}
        lists = {c: torch.empty((counts[c], 4), dtype=torch.int32, device=dev) for c in classes}
        copy = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()
        te = time.perf_counter()
        p2 = eri.Plan(s, spherical=True, schwarz_tau=1e-10, stream=stream)
        for c in classes:
            eri.eri_plan_class_quartets(p2.handle, c, 0, counts[c], lists[c], stream)
            eri.eri_compute_screened(p2.handle, c, 0, counts[c], outs[c], stream)
            done = torch.cuda.Event()
            done.record(stream)
            copy.wait_event(done)
            with torch.cuda.stream(copy):
                host[c].copy_(outs[c], non_blocking=True)
                hlist[c].copy_(lists[c], non_blocking=True)
        torch.cuda.synchronize()
        te = time.perf_counter() - te
        p2.close()
        e2e = {"value": nq * world / te, "unit": "quartets/s",
               "h2d_bytes_per_step": s.n * 48 + s.exps.size * 16, "d2h_bytes_per_step": out_bytes + nq * 16,
               "wall_s": te, "includes": "plan creation (Schwarz screen), compute, quartet lists, readback"}
        del host, hlist, lists
    cpu = None
    if rank == 0 and a.cpu_baseline:
        rate, desc, cores = cpu_oracle_rate_cluster(s, counts, budget_s=a.ref_budget)
        cpu = {"value": rate, "unit": "quartets/s", "cores": cores, "kind": "oracle", "sample": desc}
    line = {"metric": METRIC, "value": value, "unit": "quartets/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "per_class": per_class,
            "config": {"workload": wl["desc"], "unique_quartets": nq, "stored_values": out_bytes // 8,
                       "stored_bytes": out_bytes, "primitive_quartets": sum(prim_q.values()),
                       "plan_create_s": plan_s, "l2": "no flush: stored output (GBs) far exceeds L2",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "alu", "kernel": "all class kernels of the store step", "achieved": ach,
                         "peak": peak, "unit": "TFLOP/s", "frac": ach / peak, "traffic": None,
                         "peak_source": peak_src},
            "fp64_probe": probe, "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": a.steps * len(classes)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if dist:
        dist.destroy_process_group()


def cpu_oracle_rate_cluster(s, counts, budget_s=12.0):
    """Oracle quartets/s on random unique quartets of the cluster, per class,
    projected to the class mix of the screened set."""
    import oracle
    S = oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)
    rng = np.random.default_rng(5)
    by_l = {}
    for i, L in enumerate(s.L):
        by_l.setdefault(int(L), []).append(i)
    tot_q = sum(counts.values())
    classes = [c for c, n in counts.items() if n]
    share = budget_s / len(classes)
    total_time = 0.0
    done_all = 0
    for c in classes:
        spent, done, m = 0.0, 0, 16
        while spent < share:
            q = np.array([[rng.choice(by_l[l]) for l in c] for _ in range(m)], dtype=np.int32)
            t = time.perf_counter()
            oracle.eri_blocks(S, q, spherical=True)
            dt = time.perf_counter() - t
            spent += dt
            done += m
            if dt < share / 8:
                m *= 2
        total_time += spent / done * counts[c]
        done_all += done
    return tot_q / total_time, f"oracle on {done_all} random quartets over {len(classes)} classes, projected to the " \
        f"screened class mix", oracle.default_threads()


def deriv_stats(cls):
    """Generator statistics of a derivative kernel (csrc/generated/classes.json)."""
    meta = json.load(open(os.path.join(ROOT, "electron_repulsion_integrals_gb300", "csrc", "generated",
                                       "classes.json")))["classes"]["d{}{}{}{}".format(*cls)]
    return {"vrr_flops": meta["vrr_flops"], "hrr_flops": meta["hrr_flops"]}


def run_ours(a, rank, world, local_rank):
    import torch
    import electron_repulsion_integrals_gb300 as eri
    from electron_repulsion_integrals_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    eri.lib()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[a.workload]
    stream = torch.cuda.current_stream()

    # inputs resident in HBM: one plan per class batch and its quartet list
    batches = []
    for cls, n, deg, seed in wl["classes"]:
        n = max(1, int(n * a.scale))
        s, q = W.homogeneous(cls, n, deg, seed_index=seed)
        plan = eri.Plan(s, spherical=True)
        qd = torch.as_tensor(q, device=dev)
        deriv = bool(wl.get("deriv"))
        out = torch.empty(n * eri.block_size(cls) * (12 if deriv else 1), dtype=torch.float64, device=dev)
        st = eri.eri_class_info(cls)
        if deriv:
            st = dict(st, **deriv_stats(cls))
            st["staged"] = 2
        flops_q = st["vrr_flops"] * deg ** 4 + st["hrr_flops"]
        batches.append(dict(cls=cls, n=n, deg=deg, shells=s, q=q, plan=plan, qd=qd, out=out, flops=flops_q,
                            stats=st))
    torch.cuda.synchronize()
    compute = eri.eri_compute_class_deriv if wl.get("deriv") else eri.eri_compute_class

    def step(record=None):
        for b in batches:
            if record is not None:
                record[b["cls"]][0].record(stream)
            compute(b["plan"].handle, b["cls"], b["qd"], b["out"], stream)
            if record is not None:
                record[b["cls"]][1].record(stream)

    probe = measure_fp64_peak(dev, stream, local_rank)
    for _ in range(max(a.warmup, 0)):
        step()
    torch.cuda.synchronize()
    # timed region
    evs = {b["cls"]: [] for b in batches}
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(a.steps):
        rec = {b["cls"]: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for b in batches}
        step(rec)
        for k, v in rec.items():
            evs[k].append(v)
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    ms = max_over_ranks(ms, dist, dev)
    value = replica_rate(sum(b["n"] for b in batches), world, a.steps, ms)
    peak, peak_src = roofline_peak(probe, clk.get("sm_mhz"))

    per_class = {}
    for b in batches:
        kms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs[b["cls"]])
        tf = b["flops"] * b["n"] / (kms / 1e3) / 1e12
        per_class["({}{}|{}{})".format(*b["cls"])] = {
            "quartets_per_s": b["n"] / (kms / 1e3), "primitive_quartets_per_s": b["n"] * b["deg"] ** 4 / (kms / 1e3),
            "ms_per_launch": kms, "fp64_gflops": tf * 1e3, "frac_fp64_peak": tf / peak,
            "flops_per_quartet": b["flops"], "tier": ["reg", "staged", "coop"][b["stats"]["staged"]]}
    dom = max(batches, key=lambda b: b["flops"] * b["n"])
    dname = "({}{}|{}{})".format(*dom["cls"])
    ach = per_class[dname]["fp64_gflops"] / 1e3

    # end to end through the C ABI with host buffers: every step creates each
    # class's plan from host shells, copies its quartet list from pinned host
    # memory, computes, and reads all blocks back into pinned host memory.  The
    # class batches run on their own streams, heaviest first, so that one
    # batch's plan creation (host work) overlaps the other's compute and copies.
    e2e = None
    if a.e2e:
        def pinned(a):
            t = torch.empty(a.shape, dtype=torch.from_numpy(a[:0]).dtype, pin_memory=True)
            t.numpy()[...] = a
            return t.numpy()

        # the step's inputs in page-locked host memory: quartet lists and shells
        host_q = [torch.from_numpy(pinned(b["q"])) for b in batches]
        host_s = [W.Shells(*(pinned(x) for x in (b["shells"].centers, b["shells"].L, b["shells"].nprim,
                                                  b["shells"].exps, b["shells"].coefs))) for b in batches]
        host_o = [torch.empty(b["out"].numel(), dtype=torch.float64, pin_memory=True) for b in batches]
        streams = [torch.cuda.Stream() for _ in batches]
        copy_streams = [torch.cuda.Stream() for _ in batches]
        order = sorted(range(len(batches)), key=lambda i: -batches[i]["flops"] * batches[i]["n"])
        # plan creation uploads per shell its centre, l, primitive count, primitive
        # offset and first function (40 B), per primitive the exponent and coefficient
        h2d = sum(hq.numel() * 4 for hq in host_q) + sum(b["shells"].n * 40 + b["shells"].exps.size * 16
                                                         for b in batches)
        d2h = sum(ho.numel() * 8 for ho in host_o)
        e_steps = 10  # whole-run mean: one step slowed by the shared host's DMA weighs a tenth

        def e2e_step():
            plans = []
            for i in order:
                b, hq, ho, st_i, cp_i = batches[i], host_q[i], host_o[i], streams[i], copy_streams[i]
                per_q = b["out"].numel() // b["n"]
                with torch.cuda.stream(st_i):
                    plan = eri.Plan(host_s[i], spherical=True, stream=st_i)
                    qd = hq.to(dev, non_blocking=True)
                    # the chunks of one plan run in order on its stream (they
                    # share the plan's scratch); each chunk's readback runs on a
                    # copy stream, overlapping the next chunk's compute
                    for lo, hi in e2e_chunks(b["n"], b["out"].numel() * 8):
                        o = b["out"][lo * per_q:hi * per_q]
                        compute(plan.handle, b["cls"], qd[lo:hi], o, st_i)
                        done = torch.cuda.Event()
                        done.record(st_i)
                        cp_i.wait_event(done)
                        with torch.cuda.stream(cp_i):
                            ho[lo * per_q:hi * per_q].copy_(o, non_blocking=True)
                plans.append(plan)
            torch.cuda.synchronize()
            for plan in plans:
                plan.close()

        for _ in range(max(a.warmup, 3)):  # untimed: first use of the streams and of the pinned buffers
            e2e_step()
        torch.cuda.synchronize()
        steps_ms = []
        te = time.perf_counter()
        for _ in range(e_steps):
            t_s = time.perf_counter()
            e2e_step()
            steps_ms.append((time.perf_counter() - t_s) * 1e3)
        te = time.perf_counter() - te
        # value over the whole timed run (a slow host copy in one step counts); the
        # median and minimum step show the spread (the host is shared)
        e2e = {"value": sum(b["n"] for b in batches) * world * e_steps / te, "unit": "quartets/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": te / e_steps * 1e3,
               "ms_per_step_median": statistics.median(steps_ms), "ms_per_step_min": min(steps_ms),
               "ms_steps": [round(t, 1) for t in steps_ms],
               "schedule": "class batches on separate CUDA streams, heaviest first; each batch in chunks of about "
                           f"{E2E_CHUNK_BYTES / 1e9:.2g} GB of output whose readback overlaps the next chunk's compute"}

    cpu = None
    if rank == 0 and a.cpu_baseline:
        rate, desc, cores, _ = cpu_oracle_rate(wl, budget_s=a.ref_budget)
        cpu = {"value": rate, "unit": "quartets/s", "cores": cores, "kind": "oracle",
               "sample": desc + ", projected to the full step mix"}

    line = {"metric": METRIC, "value": value, "unit": "quartets/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl["desc"] + ("" if a.scale == 1 else f" (scaled x{a.scale})"),
                       "l2": "no flush: inputs and outputs of a step exceed the 126 MB L2",
                       "parallelism": f"replicas x{world}"},
            "per_class": per_class,
            "roofline": {"bound": "alu", "kernel": dname, "achieved": ach, "peak": peak,
                         "unit": "TFLOP/s", "frac": ach / peak,
                         "traffic": dram_traffic(dom["cls"], dom["n"], bool(wl.get("deriv"))),
                         "peak_source": peak_src},
            "fp64_probe": probe, "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": len(batches) * a.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)
    for b in batches:
        b["plan"].close()
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------- every class
def classes_n(fq, deg):
    """Quartets per launch of a class in the per-class table: about 8 GFLOP of
    algorithmic work, between 2,048 and 2^21 quartets."""
    return int(min(1 << 21, max(2048, 8e9 / fq)))


def run_classes(a, local_rank):
    """Every canonical class through (ff|ff) at contraction degree 1 and 2: one
    JSON line with quartets/s, FP64 GFLOP/s, fraction of the measured FP64
    peak, tier, registers and ptxas spill bytes per class, each class checked
    against the oracle on a sample."""
    import torch
    import oracle
    import electron_repulsion_integrals_gb300 as eri
    from electron_repulsion_integrals_gb300 import workloads as W
    from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    eri.lib()
    stream = torch.cuda.current_stream()
    ptx = json.load(open(os.path.join(os.path.dirname(eri.LIB_PATH), "ptxas.json")))
    probe = measure_fp64_peak(dev, stream, local_rank)
    clocks = ClockSampler(local_rank)
    clocks.start()
    rows = {}
    for cls in canonical_classes(3):
        st = eri.eri_class_info(cls)
        for deg in (1, 2):
            fq = st["vrr_flops"] * deg ** 4 + st["hrr_flops"]
            n = classes_n(fq, deg)
            s, q = W.homogeneous(cls, n, deg, seed_index=300 + 10 * sum(cls) + deg)
            plan = eri.Plan(s, spherical=True)
            qd = torch.as_tensor(q, device=dev)
            out = torch.empty(n * eri.block_size(cls), dtype=torch.float64, device=dev)
            for _ in range(max(a.warmup, 1)):
                eri.eri_compute_class(plan.handle, cls, qd, out, stream)
            evs = []
            for _ in range(a.steps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                eri.eri_compute_class(plan.handle, cls, qd, out, stream)
                e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
            idx = np.sort(np.random.default_rng(11).choice(n, 8, replace=False))
            got = out.view(n, -1)[torch.as_tensor(idx, device=dev)].cpu().numpy().ravel()
            ref = oracle.eri_blocks(oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs), q[idx],
                                    spherical=True)
            ok = bool(np.all(np.abs(got - ref) <= np.maximum(1e-12, 1e-10 * np.abs(ref))))
            # the cooperative tier is built only as its contracted instantiation
            contracted = deg > 1 or st["staged"] == 2
            kern = [k for k in ptx if "k_c{}{}{}{}I".format(*cls) in k and "ILi0E" in k
                    and ("Lb1E" in k) == contracted]
            tf = fq * n / (ms / 1e3) / 1e12
            rows["({}{}|{}{}) degree {}".format(*cls, deg)] = {
                "quartets": n, "ms_per_launch": ms, "quartets_per_s": n / (ms / 1e3),
                "primitive_quartets_per_s": n * deg ** 4 / (ms / 1e3), "fp64_gflops": tf * 1e3,
                "flops_per_quartet": fq, "tier": ["reg", "staged", "coop"][st["staged"]], "parity_ok": ok,
                "registers": max((ptx[k].get("registers", 0) for k in kern), default=None),
                "spill_bytes": max((ptx[k].get("spill_stores", 0) + ptx[k].get("spill_loads", 0) for k in kern),
                                   default=None)}
            plan.close()
            del out, qd
            torch.cuda.empty_cache()
    clk = clocks.stop()
    peak, peak_src = roofline_peak(probe, clk.get("sm_mhz"))
    for v in rows.values():
        v["frac_fp64_peak"] = v["fp64_gflops"] / 1e3 / peak
    line = {"metric": METRIC, "unit": "quartets/s", "workload": "classes", "steps": a.steps, "warmup": a.warmup,
            "dtype": "f64", "data": "synthetic", "config": {"workload": WORKLOADS["classes"]["desc"]},
            "peak": {"tflops": peak, "source": peak_src}, "fp64_probe": probe, "clocks": clk,
            "all_parity_ok": all(v["parity_ok"] for v in rows.values()), "classes": rows}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ablations
def ablation_n(cls):
    """Quartets per class in the ablation runs: outputs above L2 where the
    block allows, launches of a millisecond or more."""
    L = sum(cls)
    return {0: 1 << 22, 2: 1 << 21, 4: 1 << 20, 6: 1 << 18, 7: 1 << 17, 8: 1 << 17, 10: 1 << 15, 12: 1 << 13,
            14: 1 << 12, 16: 1 << 11}[L]


def run_ablation_worker(a):
    """One library (ERI_GB300_LIBRARY, else the main build): every class it
    holds, timed and checked against the oracle on a sample."""
    import torch
    import oracle
    import electron_repulsion_integrals_gb300 as eri
    from electron_repulsion_integrals_gb300 import workloads as W
    from electron_repulsion_integrals_gb300 import ablation
    dev = torch.device("cuda", 0)
    eri.lib()
    if a.ablation_worker == "full":
        classes = sorted(set(map(tuple, ablation.GRAPH_CLASSES + ablation.TIER_CLASSES)), key=lambda c: (sum(c), c))
    else:
        classes = ablation.VARIANTS[a.ablation_worker][0]
    stream = torch.cuda.current_stream()
    res = {}
    for cls in classes:
        n = ablation_n(cls)
        s, q = W.homogeneous(cls, n, 1, seed_index=60 + sum(cls))
        plan = eri.Plan(s, spherical=True)
        qd = torch.as_tensor(q, device=dev)
        out = torch.empty(n * eri.block_size(cls), dtype=torch.float64, device=dev)
        for _ in range(max(a.warmup, 1)):
            eri.eri_compute_class(plan.handle, cls, qd, out, stream)
        torch.cuda.synchronize()
        evs = []
        for _ in range(a.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            eri.eri_compute_class(plan.handle, cls, qd, out, stream)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
        idx = np.sort(np.random.default_rng(9).choice(n, 12, replace=False))
        got = out.view(n, -1)[torch.as_tensor(idx, device=dev)].cpu().numpy().ravel()
        ref = oracle.eri_blocks(oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs), q[idx], spherical=True)
        tol = np.maximum(1e-12, 1e-10 * np.abs(ref))
        if max(cls) >= 4:  # g shells: 1e-6 of the block maximum
            bs = ref.size // len(idx)
            tol = np.maximum(tol, 1e-6 * np.repeat(np.abs(ref).reshape(-1, bs).max(axis=1), bs))
        ok = bool(np.all(np.abs(got - ref) <= tol))
        st = eri.eri_class_info(cls)
        res["{}{}{}{}".format(*cls)] = {"quartets_per_s": n / (ms / 1e3), "ms_per_launch": ms, "quartets": n,
                                       "parity_ok": ok, "vrr_ops": st["vrr_ops"], "hrr_ops": st["hrr_ops"],
                                       "tier": ["reg", "staged", "coop"][st["staged"]]}
        plan.close()
        del out, qd
        torch.cuda.empty_cache()
    print(json.dumps(res), flush=True)


def run_ablation(a):
    """Each ablation library against the main build, class by class."""
    import subprocess
    import electron_repulsion_integrals_gb300 as eri
    from electron_repulsion_integrals_gb300 import ablation
    names = a.ablation.split(",") if a.ablation != "all" else list(ablation.VARIANTS)
    t = time.perf_counter()
    paths = ablation.build_all(names)
    build_s = time.perf_counter() - t
    out = {"metric": "ablation: quartets/s per class and library (FusionRCG section V-B switches)", "unit": "quartets/s",
           "steps": a.steps, "warmup": a.warmup, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "per class: homogeneous batch, degree 1, centers U[0,10]^3 bohr, exponents "
                                  "log-U[0.05,100], spherical; quartets per class by total angular momentum"},
           "build_s": build_s, "libraries": {}}
    for name in ["full"] + names:
        env = dict(os.environ)
        if name != "full":
            env["ERI_GB300_LIBRARY"] = paths[name]
        cmd = [sys.executable, os.path.abspath(__file__), "--ablation-worker", name, "--steps", str(a.steps),
               "--warmup", str(a.warmup)]
        r = subprocess.run(cmd, env=env, capture_output=True, text=True)
        if r.returncode != 0:
            out["libraries"][name] = {"error": r.stderr[-2000:]}
            continue
        res = json.loads(r.stdout.strip().splitlines()[-1])
        meta = {}
        if name != "full":
            cj = json.load(open(os.path.join(os.path.dirname(paths[name]), "classes.json")))
            meta = cj["classes"]
            ptx = json.load(open(os.path.join(os.path.dirname(paths[name]), "ptxas.json")))
        else:
            meta = json.load(open(os.path.join(ROOT, "electron_repulsion_integrals_gb300", "csrc", "generated",
                                               "classes.json")))["classes"]
            meta = {"{}{}{}{}".format(*m["cls"]) if isinstance(m, dict) and "cls" in m else k: m
                    for k, m in (meta.items() if isinstance(meta, dict) else enumerate(meta))}
            ptx = json.load(open(os.path.join(os.path.dirname(eri.LIB_PATH), "ptxas.json")))
        for c, v in res.items():
            m = meta.get(c, {})
            v.update({k: m.get(k) for k in ("peak_live", "schedule", "rule", "shape", "sph_fusion", "arena")
                      if k in m})
            kern = [k for k in ptx if f"k_c{c}I" in k and "ILi0E" in k]
            if kern:
                v["registers"] = max(ptx[k].get("registers", 0) for k in kern)
                v["spill_bytes"] = max(ptx[k].get("spill_stores", 0) + ptx[k].get("spill_loads", 0) for k in kern)
        out["libraries"][name] = res
    full = out["libraries"].get("full", {})
    out["speedup_vs_full"] = {name: {c: v["quartets_per_s"] / full[c]["quartets_per_s"]
                                     for c, v in lib.items() if c in full and "quartets_per_s" in v}
                              for name, lib in out["libraries"].items() if name != "full" and "error" not in lib}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="homogeneous", choices=sorted(WORKLOADS))
    ap.add_argument("--scale", type=float, default=1.0, help="fraction of the workload's quartets (profiling)")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work per sample")
    ap.add_argument("--ablation", default=None, help="'all' or comma-separated ablation libraries to time")
    ap.add_argument("--ablation-worker", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--fp64-peak", action="store_true", help="sweep the FP64 rate probe and print its rates")
    a = ap.parse_args()
    if a.ablation_worker:
        run_ablation_worker(a)
        return
    if a.ablation:
        run_ablation(a)
        return
    if a.fp64_peak:
        if env_int("RANK", 0) == 0:
            run_fp64_peak(a, env_int("LOCAL_RANK", 0))
        return
    rank = env_int("RANK", 0)
    world = env_int("WORLD_SIZE", 1)
    local_rank = env_int("LOCAL_RANK", 0)
    if a.impl == "reference":
        run_reference(a, rank, world)
    elif a.workload == "classes":
        if rank == 0:
            run_classes(a, local_rank)
    elif WORKLOADS[a.workload].get("store"):
        run_store(a, rank, world, local_rank)
    elif "cluster" in WORKLOADS[a.workload]:
        run_coulomb(a, rank, world, local_rank)
    else:
        run_ours(a, rank, world, local_rank)


if __name__ == "__main__":
    main()
