"""Benchmark of the DFlash 2 draft-block head on GB300.

One step = one full draft-verify cycle of the head over a batch of sequences
(the whole hot path): two-tap dynamic conv x10 (each application on its own
activation, the last one feeding the gate) -> top-16 -> context gate + pair
scores -> walk (T=0) -> verify (T=0) -> walk (T=1) -> verify (T=1), on seeded
synthetic inputs of the pages' shapes (B=128, L=16, V=151936, d=5120).

Prints ONE JSON line (rank 0).  `value` is draft blocks per second with the
inputs resident in HBM; `e2e` is the same metric through the public API with
host (pinned) buffers, host<->device copies inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dflash2|reference]
                  [--no-sweep] [--no-e2e] [--no-cpu-baseline] [--no-lmhead] [--no-next]
                  [--no-small]

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload instead.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from draft_selection_dflash2_gb300 import replicas, synth  # noqa: E402

METRIC = "draft blocks/s"
UNIT = "blocks/s"
B, L, V, D, R, K = 128, 16, 151936, 5120, 256, 16
CONV_APPS = 10
WORKLOAD = (f"full draft-verify cycle B={B} L={L} V={V} d={D}: two-tap conv x{CONV_APPS} (each on its own "
            "[B,L,d] activation), top-16, gate + pair scores, walk T=0 and T=1, verify T=0 and T=1")
PAIRS_PER_BLOCK = K + K * K * (L - 1)   # 16 at t=0 (one predecessor), 256 per later position
SWEEP_B = (1, 8, 32, 128, 256)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# algorithmic bytes per stage (what the method must move, not what a kernel does)
# ---------------------------------------------------------------------------
def bytes_topk(nb):
    return nb * L * V * 2 + nb * L * K * 8


def bytes_pairs(nb):
    per_block = L * D * 2 + (K * (L - 1) + 1) * R * 2 + K * L * R * 2 + L * K * K * 4 + L * K * 8
    return nb * per_block + R * D * 2


def bytes_conv(nb):
    return nb * L * D * 2 * 2 + nb * D * 2 + 2 * (D // 16) * D * 2 + 2 * D * 2


def bytes_verify(acc):
    return int(np.sum(acc.astype(np.int64))) * V * 2


def bytes_walk(nb):
    return nb * L * K * K * 4 + nb * L * K * 4


# ---------------------------------------------------------------------------
# DRAM traffic per launch from the committed ncu summaries, valid only while
# the kernel's sources are unchanged since the capture (else null)
# ---------------------------------------------------------------------------
_CSRC = os.path.join(ROOT, "draft_selection_dflash2_gb300", "csrc")
_PROFILED = {
    "conv": ["conv2tap_B128_d5120.md"],
    "topk": ["topk16_B128_V151936.md"],
    "pairs": ["gate_gemm_B128_d5120.md", "pair_kernel_B128.md"],
    "verify0": ["verify_kernel_T0_B128.md"],
    "verify1": ["verify_kernel_T1_B128.md"],
    "walk0": ["walk_T0_B128.md"],
    "walk1": ["walk_T1_B128.md"],
}
_SOURCES = {
    "topk16": ["topk.cu", "common.cuh"],
    "conv2tap": ["conv2tap.cu", "gemm_pair.cuh", "tcgen05.cuh", "common.cuh"],
    "verify": ["verify.cu", "common.cuh", "philox.cuh"],
    "pair_scores": ["select.cu", "gemm_pair.cuh", "tcgen05.cuh", "common.cuh"],
    "proj": ["proj.cu", "pair_math.cuh", "tcgen05.cuh", "common.cuh"],
    "walk": ["walk.cu", "common.cuh", "philox.cuh", "exp2.cuh"],
    "lmhead": ["lmhead.cu", "tcgen05.cuh", "common.cuh"],
    "viterbi": ["viterbi.cu", "common.cuh"],
    "eval": ["eval.cu", "common.cuh"],
    "gemm_conv": ["gemm_conv.cu", "tcgen05.cuh", "common.cuh"],
}
_PROFILE_SOURCES = {"conv2tap_B128_d5120.md": "conv2tap", "topk16_B128_V151936.md": "topk16",
                    "gate_gemm_B128_d5120.md": "pair_scores", "pair_kernel_B128.md": "pair_scores",
                    "verify_kernel_T0_B128.md": "verify", "verify_kernel_T1_B128.md": "verify",
                    "walk_T0_B128.md": "walk", "walk_T1_B128.md": "walk", "lmhead_M1024_V151936_d5120.md": "lmhead",
                    "walk_viterbi_B16384.md": "viterbi", "selector_eval_B524288.md": "eval",
                    "proj_kernel_B128_d5120.md": "proj", "gemm_conv_kernel_B128_K5120_d5120.md": "gemm_conv"}


def _source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in _SOURCES[kernel]:
        with open(os.path.join(_CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(names):
    """Sum of dram bytes per launch over the named summaries, or None if any is
    missing or was captured from different kernel sources."""
    total = 0
    for name in names:
        path = os.path.join(ROOT, "profiles", name)
        if not os.path.exists(path):
            return None
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.split(":")[0] in ("dram-bytes-per-launch", "source-sha256"):
                    k, v = line.split(":", 1)
                    fields[k] = v.strip()
        if fields.get("source-sha256") != _source_hash(_PROFILE_SOURCES[name]):
            return None
        total += int(fields["dram-bytes-per-launch"])
    return total


# ---------------------------------------------------------------------------
# clocks sampled with nvidia-smi during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, torch):
        self.proc = None
        self.path = os.path.join("/tmp", f"dflash2_clocks_{os.getpid()}.csv")
        try:
            p = torch.cuda.get_device_properties(torch.cuda.current_device())
            self.sel = ["-i", f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"]
        except Exception:
            self.sel = []

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 6:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[2:6]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def make_host_workload(nb, sweep_rows=0, rank=0):
    """Seeded host tensors of the full-cycle workload (bf16 as uint16 bits).
    Per-sequence data depends on the rank (each replica drafts its own batch);
    the parameters (conv kernels, W_H, A, B) are shared."""
    sd = lambda s: replicas.rank_seed(s, rank)  # noqa: E731
    rng = np.random.default_rng(sd(0))
    rows = max(nb * L, sweep_rows)
    w = {}
    w["U"] = synth.logits_planted(rng, rows, V)
    # each conv application reads its own activation (in the drafter every
    # sublayer boundary presents a new hidden state), so nothing is chained
    w["conv"] = [(synth.normal_bits(sd(100 + a), (nb, L, D)), synth.normal_bits(sd(200 + a), (nb, D)))
                 + synth.conv_layer_params(10 + a, D) for a in range(CONV_APPS)]
    w["W_H"] = synth.normal_bits(3, (R, D), std=0.02)
    w["A"] = synth.normal_bits(4, (V, R), std=0.02)
    w["Bt"] = synth.normal_bits(5, (V, R), std=0.02)
    w["last_verified"] = np.random.default_rng(sd(6)).integers(0, V, nb).astype(np.int32)
    return w


def to_dev(torch, a, dev):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else np.ascontiguousarray(a))
    t = t.to(dev)
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


LEAD_CYCLES = 4_000_000   # ~2 ms of device clock at 2 GHz


def device_lead(torch):
    """Queue a device-side wait (a clock spin of LEAD_CYCLES) ahead of a timed
    region, so that the host has enqueued the timed launches before the first
    event fires: the events then time the device's work, not the host's launch
    latency.  The wait itself lies before the first event."""
    torch.cuda._sleep(LEAD_CYCLES)


class Cycle:
    """Device buffers and the step of the full cycle, through the Python API."""

    def __init__(self, torch, api, h, w, nb, dev):
        self.torch, self.api, self.h, self.nb = torch, api, h, nb
        bf = lambda a: to_dev(torch, a, dev)  # noqa: E731
        self.U = bf(w["U"][: nb * L])
        self.conv = [(bf(x), bf(xp), bf(k0), bf(k1), bf(W)) for x, xp, k0, k1, W in w["conv"]]
        self.W_H, self.A, self.Bt = bf(w["W_H"]), bf(w["A"]), bf(w["Bt"])
        self.lv = to_dev(torch, w["last_verified"], dev)
        self.ybuf = [torch.empty((nb, L, D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.vals = torch.empty((nb * L, K), dtype=torch.float32, device=dev)
        self.idx = torch.empty((nb * L, K), dtype=torch.int32, device=dev)
        self.gate = torch.empty((nb, L, R), dtype=torch.float32, device=dev)
        self.S = torch.empty((nb, L, K, K), dtype=torch.float32, device=dev)
        self.tok = [torch.empty((nb, L), dtype=torch.int32, device=dev) for _ in range(2)]
        self.slot = [torch.empty((nb, L), dtype=torch.int32, device=dev) for _ in range(2)]
        self.q = [torch.empty((nb, L, K), dtype=torch.float32, device=dev) for _ in range(2)]
        self.acc = [torch.empty((nb,), dtype=torch.int32, device=dev) for _ in range(2)]
        self.out = [torch.empty((nb, L + 1), dtype=torch.int32, device=dev) for _ in range(2)]
        self.target = None
        self.vws = torch.empty(api.verify_workspace(h, nb, L, V), dtype=torch.uint8, device=dev)
        self.cws = torch.empty(api.conv2tap_workspace(h, nb, L, D), dtype=torch.uint8, device=dev)
        self.pws = torch.empty(api.pair_scores_workspace(h, nb, L, D), dtype=torch.uint8, device=dev)
        # conv x10 (pair GEMM + tap kernel each), top-16, gate GEMM + pair kernel, walk and verify at T=0
        # (init + greedy kernel) and T=1 (init + rows kernel + draw kernel)
        self.launches_per_step = 2 * CONV_APPS + 1 + 2 + (1 + 2) + (1 + 3)

    def step(self, ev=None, seed_offset=0):
        api, h = self.api, self.h
        rec = (lambda name: ev[name].record()) if ev else (lambda name: None)
        rec("start")
        for a, (x, xp, k0, k1, W) in enumerate(self.conv):
            cur = api.conv2tap(h, x, xp, k0, k1, W, y=self.ybuf[a % 2], workspace=self.cws)
        rec("conv")
        api.topk(h, self.U, vals=self.vals, idx=self.idx)
        rec("topk")
        ci, cv = self.idx.view(self.nb, L, K), self.vals.view(self.nb, L, K)
        api.pair_scores(h, ci, cv, self.lv, cur, self.W_H, None, self.A, self.Bt, gate=self.gate, S=self.S,
                        workspace=self.pws)
        rec("pairs")
        for i, T in enumerate((0.0, 1.0)):
            api.walk(h, self.S, ci, temperature=T, seed=1, offset=seed_offset, draft_tok=self.tok[i],
                     draft_slot=self.slot[i], draft_q=self.q[i])
            rec(f"walk{i}")
            api.verify(h, self.target, self.tok[i], self.slot[i], self.q[i], ci, temperature=T, seed=1,
                       offset=seed_offset, accept_len=self.acc[i], out_tok=self.out[i], workspace=self.vws)
            rec(f"verify{i}")


STAGES = ["conv", "topk", "pairs", "walk0", "verify0", "walk1", "verify1"]


def run_gpu(args):
    import torch

    from draft_selection_dflash2_gb300 import api, build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        build.build()
    if dist:
        dist.barrier()
    build.build()
    pk = peaks()
    h = api.Handle(torch.cuda.current_device())

    sweep_rows = max(SWEEP_B) * L if (args.sweep and rank == 0) else 0
    w = make_host_workload(B, sweep_rows, rank)
    cyc = Cycle(torch, api, h, w, B, dev)
    # plant the target on the greedy draft of one untimed cycle: 0.85 argmax agreement
    cyc.target = torch.empty((B, L + 1, V), dtype=torch.bfloat16, device=dev)
    cyc.step()
    torch.cuda.synchronize()
    draft = cyc.tok[0].cpu().numpy()
    tgt = synth.target_planted(replicas.rank_seed(7, rank), draft, V, agree=0.85, plant=8.0)
    cyc.target.copy_(to_dev(torch, tgt, dev))
    stream = torch.cuda.current_stream()

    for i in range(args.warmup):
        cyc.step(seed_offset=i)
    torch.cuda.synchronize()
    assert h.device_error() == 0, "device error during warm-up"

    # timed region
    evs = [{n: torch.cuda.Event(enable_timing=True) for n in ["start"] + STAGES} for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    device_lead(torch)
    t0.record(stream)
    host0 = time.perf_counter()
    for i in range(args.steps):
        cyc.step(seed_offset=1000 + i)
    host_ms = (time.perf_counter() - host0) * 1e3 / args.steps
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    elapsed_ms = replicas.max_over_ranks(t0.elapsed_time(t1), dist, dev)
    assert h.device_error() == 0, "device error during the timed region"
    # the stage breakdown: the same steps again with an event between stages (an
    # event between two kernels stops the next one from starting early, so the
    # timed pass above records none)
    device_lead(torch)
    for i in range(args.steps):
        cyc.step(ev=evs[i], seed_offset=1000 + i)
    torch.cuda.synchronize()

    stage_ms = {}
    for n in STAGES:
        prev = ["start"] + STAGES
        p = prev[prev.index(n) - 1]
        stage_ms[n] = statistics.median(evs[i][p].elapsed_time(evs[i][n]) for i in range(args.steps))
    acc0 = cyc.acc[0].cpu().numpy()
    acc1 = cyc.acc[1].cpu().numpy()

    value = replicas.whole_job_rate(B * args.steps, world, elapsed_ms / 1e3)
    ms_per_step = elapsed_ms / args.steps
    hbm = pk["hbm_gbs"]
    stage_bytes = {"conv": CONV_APPS * bytes_conv(B), "topk": bytes_topk(B), "pairs": bytes_pairs(B),
                   "walk0": bytes_walk(B), "verify0": bytes_verify(acc0), "walk1": bytes_walk(B),
                   "verify1": bytes_verify(acc1)}
    stages = {}
    for n in STAGES:
        gbs = stage_bytes[n] / (stage_ms[n] * 1e-3) / 1e9
        stages[n] = {"ms": round(stage_ms[n], 4), "alg_bytes": stage_bytes[n], "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / hbm, 4)}
    stages["conv"]["per_application_ms"] = round(stage_ms["conv"] / CONV_APPS, 4)
    dom = max(STAGES, key=lambda n: stage_ms[n])
    kernel_name = {"conv": "pair_gemm_kernel<ConvShape> + conv_tap_kernel", "topk": "topk16_kernel",
                   "pairs": "pair_gemm_kernel<GateShape> + pair_kernel",
                   "walk0": "walk_kernel", "walk1": "walk_kernel", "verify0": "verify_greedy_kernel",
                   "verify1": "verify_rows_kernel + verify_draw_kernel"}[dom]
    per_launch_ms = stage_ms[dom] / (CONV_APPS if dom == "conv" else 1)
    per_launch_bytes = stage_bytes[dom] / (CONV_APPS if dom == "conv" else 1)
    achieved = per_launch_bytes / (per_launch_ms * 1e-3) / 1e9
    traffic = profiled_traffic(_PROFILED[dom]) if dom in _PROFILED else None
    roofline = {"bound": "hbm", "kernel": kernel_name, "stage": dom, "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": traffic, "traffic_unit": "bytes per launch (ncu, profiles/)",
                "alg_bytes_per_launch": int(per_launch_bytes),
                "peak_source": pk["source"] + " (burst copy, MEASURED_PEAKS.json)"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate (fp64 sampling decisions)",
        "data": "synthetic (seeded; shapes of the pages' workloads, no datasets or trained weights)",
        "config": {"workload": WORKLOAD, "B": B, "L": L, "V": V, "d": D, "K": K, "r": R,
                   "conv_applications": CONV_APPS, "parallelism": f"replicas x{world} (batch-sharded)",
                   "l2": "inputs larger than L2 (622 MB logits + 661 MB target logits per step)"},
        "pair_scores_per_s": round(B * PAIRS_PER_BLOCK / (stage_ms["pairs"] * 1e-3), 1),
        "mean_accept_len": {"T0": round(float(acc0.mean()), 4), "T1": round(float(acc1.mean()), 4)},
        "stages": stages,
        "stages_pass": "per-stage CUDA events from a second pass of the same steps; their sum exceeds ms_per_step "
                       "because an event between stages stops the next kernel from overlapping the previous one",
        "roofline": roofline,
        "clocks": clk,
        "gpu_launches": cyc.launches_per_step * args.steps,
        "host_enqueue_ms_per_step": round(host_ms, 4),
        "timing": "CUDA events on the launching stream; a device-side wait queued before the first event lets "
                  "the host enqueue ahead, so the interval is the device's (host_enqueue_ms_per_step below "
                  "ms_per_step: the device never waited for the host)",
    }

    if rank == 0 and args.sweep:
        line["sweep"] = run_sweep(torch, api, h, w, cyc, dev, pk)
        line["sweep_zipf"] = run_sweep(torch, api, h, w, cyc, dev, pk, logits="zipf")
    if rank == 0 and args.small:
        line["small_cycles"] = run_small_cycles(torch, api, h, dev)
    if rank == 0 and args.e2e:
        line["e2e"] = run_e2e(torch, api, h, w, cyc, dev, args)
    if rank == 0 and args.lmhead:
        line["lmhead"] = run_lmhead(torch, api, h, dev, pk)
    if rank == 0 and args.next:
        line["next"] = run_next(torch, api, h, cyc, dev, pk)
        line["next"]["projection_selector"]["table_form_pairs_ms_in_step"] = stages["pairs"]["ms"]
    if rank == 0 and args.cpu_baseline and world == 1:
        line["cpu_baseline"] = run_cpu_baseline(w, tgt)
    if rank == 0:
        print(json.dumps(line), flush=True)
    h.close()
    if dist:
        dist.destroy_process_group()


def _zipf_logits_dev(torch, rows, dev, seed=41):
    """Zipf(1.1)-ranked logits drawn on the device with the same recipe as
    synth.logits_zipf (N(0, 2^2) + a shared -1.1 ln(1 + rank) bias), bf16 [rows, V]."""
    bias = torch.from_numpy(synth.zipf_bias(np.random.default_rng(seed), V)).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    U = torch.empty((rows, V), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, rows, 512):
        r1 = min(rows, r0 + 512)
        U[r0:r1] = (torch.randn((r1 - r0, V), generator=g, device=dev) * 2.0 + bias).to(torch.bfloat16)
    return U


def run_sweep(torch, api, h, w, cyc, dev, pk, logits="planted"):
    """Batch sweep at d=5120: top-16 + pair scores + greedy walk, blocks/s and GB/s
    per stage, on the planted logits or on Zipf(1.1)-ranked ones."""
    out = []
    if logits == "planted":
        Ufull = to_dev(torch, w["U"][: max(SWEEP_B) * L], dev)
    else:
        Ufull = _zipf_logits_dev(torch, max(SWEEP_B) * L, dev)
    hs_all = torch.empty((max(SWEEP_B), L, D), dtype=torch.bfloat16, device=dev)
    hs_all.copy_(cyc.ybuf[1][:1].expand(max(SWEEP_B), L, D))
    lv = torch.zeros((max(SWEEP_B),), dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for nb in SWEEP_B:
        U = Ufull[: nb * L]
        vals = torch.empty((nb * L, K), dtype=torch.float32, device=dev)
        idx = torch.empty((nb * L, K), dtype=torch.int32, device=dev)
        gate = torch.empty((nb, L, R), dtype=torch.float32, device=dev)
        S = torch.empty((nb, L, K, K), dtype=torch.float32, device=dev)
        tok = torch.empty((nb, L), dtype=torch.int32, device=dev)
        slot = torch.empty((nb, L), dtype=torch.int32, device=dev)
        pws = torch.empty(max(api.pair_scores_workspace(h, nb, L, D), 256), dtype=torch.uint8, device=dev)
        times = {"topk": [], "pairs": [], "walk": []}
        steps = 20
        for it in range(steps + 3):
            flush.zero_()   # L2 flush (buffer larger than L2)
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            device_lead(torch)
            e[0].record()
            api.topk(h, U, vals=vals, idx=idx)
            e[1].record()
            api.pair_scores(h, idx.view(nb, L, K), vals.view(nb, L, K), lv[:nb], hs_all[:nb], cyc.W_H, None,
                            cyc.A, cyc.Bt, gate=gate, S=S, workspace=pws)
            e[2].record()
            api.walk(h, S, idx.view(nb, L, K), draft_tok=tok, draft_slot=slot, want_q=False)
            e[3].record()
            torch.cuda.synchronize()
            if it >= 3:
                times["topk"].append(e[0].elapsed_time(e[1]))
                times["pairs"].append(e[1].elapsed_time(e[2]))
                times["walk"].append(e[2].elapsed_time(e[3]))
        med = {k: statistics.median(v) for k, v in times.items()}
        tot = sum(med.values())
        # steady state: back-to-back top-16 calls over distinct rows (each call still reads rows
        # no other call read), which spreads the launch and ramp a single call pays over the calls
        nsl = min(8, Ufull.shape[0] // (nb * L))
        b2b = []
        if nsl >= 2:
            for it in range(8):
                flush.zero_()
                device_lead(torch)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for j in range(nsl):
                    api.topk(h, Ufull[j * nb * L:(j + 1) * nb * L], vals=vals, idx=idx)
                b.record()
                torch.cuda.synchronize()
                if it >= 3:
                    b2b.append(a.elapsed_time(b) / nsl)
        out.append({"B": nb, "logits": "planted N(0,1)+4" if logits == "planted" else "zipf(1.1) N(0,4)+bias",
                    "blocks_per_s": round(nb / (tot * 1e-3), 1), "ms": round(tot, 4),
                    "pair_scores_per_s": round(nb * PAIRS_PER_BLOCK / (med["pairs"] * 1e-3), 1),
                    "topk_GBps": round(bytes_topk(nb) / (med["topk"] * 1e-3) / 1e9, 1),
                    "pairs_GBps": round(bytes_pairs(nb) / (med["pairs"] * 1e-3) / 1e9, 1),
                    "topk_frac_hbm": round(bytes_topk(nb) / (med["topk"] * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                    "pairs_frac_hbm": round(bytes_pairs(nb) / (med["pairs"] * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                    "walk_us": round(med["walk"] * 1e3, 2)})
        if b2b:
            mb = statistics.median(b2b)
            out[-1]["topk_back_to_back"] = {"calls": nsl, "ms_per_call": round(mb, 4),
                                            "frac_hbm": round(bytes_topk(nb) / (mb * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}
    del flush, Ufull
    return out


def _small_inputs(torch, wl, dev):
    """Device inputs of one cycle of a small workload (seeded, synth recipes)."""
    si = synth.selector_inputs(31, wl.B, wl.L, wl.V, wl.d, logits=wl.logits)
    bf = lambda a: to_dev(torch, a, dev)  # noqa: E731
    t = {"U": bf(si.U.reshape(wl.B * wl.L, wl.V)), "W_H": bf(si.W_H), "A": bf(si.A), "Bt": bf(si.Bt),
         "lv": to_dev(torch, si.last_verified, dev)}
    if wl.conv_apps:
        c = synth.conv_inputs(32, wl.B, wl.L, wl.d)
        t.update(x=bf(c.x), xp=bf(c.x_prev), k0=bf(c.k0), k1=bf(c.k1), W_c=bf(c.W_c))
    else:
        t["hs"] = bf(si.h)
    return t


def run_small_cycles(torch, api, h, dev):
    """Microseconds per cycle at B=1 for the tiny selector (L=8, V=4096, d=512:
    top-16, gate + pair scores, walk T=0) and the Qwen3-4B-shaped head (L=16,
    V=151936, d=2560, Zipf logits: conv, top-16, gate + pair scores, walk T=0
    and T=1).  Each cycle is replayed from a CUDA graph, cycles back to back on
    one stream.  Hot L2: the same inputs every cycle.  Cold L2: the graph
    rotates through copies of all inputs and parameters whose bytes read per
    cycle add up to at least four times the L2 between two uses of a copy."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for key, wl in (("tiny_selector", synth.TINY_SELECTOR), ("qwen3_4b_head", synth.QWEN3_4B_HEAD)):
        nb, Lw, d = wl.B, wl.L, wl.d
        base = _small_inputs(torch, wl, dev)
        read = nb * Lw * wl.V * 2 + nb * Lw * d * 2 + R * d * 2 + nb * ((K * (Lw - 1) + 1) + K * Lw) * R * 2
        if wl.conv_apps:
            read += nb * d * 2 + 2 * (d // 16) * d * 2 + 2 * d * 2
        n_copies = int(min(2048, max(2, -(-4 * l2 // read))))
        copies = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(n_copies - 1)]
        vals = torch.empty((nb * Lw, K), dtype=torch.float32, device=dev)
        idx = torch.empty((nb * Lw, K), dtype=torch.int32, device=dev)
        hs = torch.empty((nb, Lw, d), dtype=torch.bfloat16, device=dev)
        gate = torch.empty((nb, Lw, R), dtype=torch.float32, device=dev)
        S = torch.empty((nb, Lw, K, K), dtype=torch.float32, device=dev)
        nT = len(wl.temperatures)
        tok = [torch.empty((nb, Lw), dtype=torch.int32, device=dev) for _ in range(nT)]
        slot = [torch.empty((nb, Lw), dtype=torch.int32, device=dev) for _ in range(nT)]
        q = [torch.empty((nb, Lw, K), dtype=torch.float32, device=dev) for _ in range(nT)]
        cws = torch.empty(max(api.conv2tap_workspace(h, nb, Lw, d), 256), dtype=torch.uint8, device=dev)
        pws = torch.empty(max(api.pair_scores_workspace(h, nb, Lw, d), 256), dtype=torch.uint8, device=dev)
        launches = (2 if wl.conv_apps else 0) + 1 + 2 + nT

        def cycle(c):
            cur = c["hs"] if "hs" in c else api.conv2tap(h, c["x"], c["xp"], c["k0"], c["k1"], c["W_c"], y=hs,
                                                         workspace=cws)
            api.topk(h, c["U"], vals=vals, idx=idx)
            ci, cv = idx.view(nb, Lw, K), vals.view(nb, Lw, K)
            api.pair_scores(h, ci, cv, c["lv"], cur, c["W_H"], None, c["A"], c["Bt"], gate=gate, S=S, workspace=pws)
            for i, T in enumerate(wl.temperatures):
                api.walk(h, S, ci, temperature=T, seed=1, draft_tok=tok[i], draft_slot=slot[i], draft_q=q[i])

        for c in copies:
            cycle(c)
        torch.cuda.synchronize()
        # eager launches from Python (host launch overhead included), hot inputs
        eager_n = 200
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(eager_n):
            cycle(copies[0])
        e1.record()
        torch.cuda.synchronize()
        eager_us = e0.elapsed_time(e1) * 1e3 / eager_n
        hot_n = 64
        g_hot, g_cold = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_hot):
            for _ in range(hot_n):
                cycle(copies[0])
        with torch.cuda.graph(g_cold):
            for c in copies:
                cycle(c)

        def per_cycle_us(g, n_cycles, reps):
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            device_lead(torch)
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) * 1e3 / (reps * n_cycles)

        hot_us = per_cycle_us(g_hot, hot_n, 20)
        cold_us = per_cycle_us(g_cold, n_copies, max(2, 2048 // n_copies))
        assert h.device_error() == 0, f"device error in the {key} cycles"
        out[key] = {"workload": wl.name + ", " + ", ".join(
                        (["conv x1"] if wl.conv_apps else []) + ["top-16", "gate + pair scores"]
                        + [f"walk T={T:g}" for T in wl.temperatures]),
                    "us_per_cycle_hot_l2": round(hot_us, 2), "us_per_cycle_cold_l2": round(cold_us, 2),
                    "us_per_cycle_eager_launch_hot_l2": round(eager_us, 2),
                    "kernel_launches_per_cycle": launches,
                    "cold_l2": f"{n_copies} rotating copies of every input and parameter, "
                               f"{read} bytes read per cycle ({n_copies * read / l2:.1f}x L2 between reuses)",
                    "timing": "CUDA graph replay, cycles back to back on one stream, CUDA events"}
        del g_hot, g_cold, copies, base
    return out


def run_lmhead(torch, api, h, dev, pk, M=1024):
    """Fused LM head + top-16 on hidden [1024, 5120] x W [151936, 5120] (bf16,
    N(0,1) and N(0,0.02), drawn on the device with a seeded torch generator),
    against the unfused library path: cuBLAS bf16 GEMM writing the logits, then
    dflash2_topk over them (timing comparison only)."""
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    hidden = torch.randn((M, D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn((V, D), generator=g, device=dev, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    ws = torch.empty(max(api.lmhead_topk_workspace(h, M, V, D), 256), dtype=torch.uint8, device=dev)
    vals = torch.empty((M, K), dtype=torch.float32, device=dev)
    idx = torch.empty((M, K), dtype=torch.int32, device=dev)
    flops = 2.0 * M * V * D

    def timed(fn):
        return _timed(torch, fn)

    fused_ms = timed(lambda: api.lmhead_topk(h, hidden, W, vals=vals, idx=idx, workspace=ws))
    W_H = (torch.randn((R, D), generator=g, device=dev, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    gate = torch.empty((M, R), dtype=torch.float32, device=dev)
    gate_ms = timed(lambda: api.lmhead_topk_gate(h, hidden, W, W_H, vals=vals, idx=idx, gate=gate, workspace=ws))
    logits = torch.empty((M, V), dtype=torch.bfloat16, device=dev)
    unfused_ms = timed(lambda: (torch.matmul(hidden, W.t(), out=logits), api.topk(h, logits, vals=vals, idx=idx)))
    tf = flops / (fused_ms * 1e-3) / 1e12
    del logits, W, hidden
    return {"workload": f"fused LM-head top-16 M={M} d={D} V={V}", "fused_ms": round(fused_ms, 4),
            "traffic": profiled_traffic(["lmhead_M1024_V151936_d5120.md"]),
            "unfused_cublas_plus_topk_ms": round(unfused_ms, 4),
            "with_gate_folded_ms": round(gate_ms, 4),
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tf / pk["bf16_tflops"], 4),
                         "peak_source": pk["source"] + " (bf16 burst, MEASURED_PEAKS.json)"}}


def _timed(torch, fn, reps=5, warm=2):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        device_lead(torch)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def _scaled_traffic(name, factor):
    """DRAM bytes of a smaller captured case scaled by the units processed (the
    traffic of these streaming kernels grows in proportion), or None."""
    t = profiled_traffic([name])
    return None if t is None else int(t * factor)


def table1_recalls():
    """Table 1's recall@1 / recall@16 per draft position, from the golden fixture."""
    rows = {}
    with open(os.path.join(ROOT, "tests", "golden", "table1_recall.txt")) as f:
        for line in f:
            parts = line.split()
            if parts and not line.startswith("#"):
                rows[parts[0]] = [float(x) for x in parts[1:8]]
    return rows["recall@1"], rows["recall@16"]


def run_next(torch, api, h, cyc, dev, pk, B_vit=65536, B_eval=1 << 21):
    """The next rows, timed beside the step (not part of it).
    viterbi: the exact best-path walk on the step's pair scores S [B, 16, 16, 16]
      (L2 flushed before each launch), and at B = 65536 on N(0, 4) scores
      (1 GiB of S: larger than L2).
    selector_eval: the Table 1 evaluation over 2^21 sequences of 7 positions with
      Table 1's recalls planted independently per position (0.9 GiB of candidate
      ids: larger than L2)."""
    g = torch.Generator(device=dev)
    g.manual_seed(17)
    out = {}
    nb = cyc.nb
    tok = torch.empty((nb, L), dtype=torch.int32, device=dev)
    slot = torch.empty((nb, L), dtype=torch.int32, device=dev)
    sc = torch.empty((nb,), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    ci = cyc.idx.view(nb, L, K)
    ms_small = _timed(torch, lambda: (flush.zero_(), api.walk_viterbi(h, cyc.S, ci, draft_tok=tok, draft_slot=slot,
                                                                      score=sc)), reps=9)
    ms_flush = _timed(torch, lambda: flush.zero_(), reps=9)
    del flush
    S = torch.randn((B_vit, L, K, K), generator=g, device=dev, dtype=torch.float32) * 2
    cidx = torch.randint(0, V, (B_vit, L, K), generator=g, device=dev, dtype=torch.int32)
    tok = torch.empty((B_vit, L), dtype=torch.int32, device=dev)
    slot = torch.empty((B_vit, L), dtype=torch.int32, device=dev)
    sc = torch.empty((B_vit,), dtype=torch.float32, device=dev)
    ms = _timed(torch, lambda: api.walk_viterbi(h, S, cidx, draft_tok=tok, draft_slot=slot, score=sc))
    nbytes = B_vit * L * (K * K * 4 + K * 4 + 8) + B_vit * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["viterbi"] = {"workload": f"B={nb} L={L} (the step's S, L2 flushed)",
                      "us": round(max(ms_small - ms_flush, 0.0) * 1e3, 2),
                      "throughput": {"workload": f"B={B_vit} L={L}", "ms": round(ms, 4),
                                     "sequences_per_s": round(B_vit / (ms * 1e-3), 1),
                                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                                                  "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                                                  "traffic": _scaled_traffic("walk_viterbi_B16384.md", B_vit / 16384),
                                                  "alg_bytes_per_launch": nbytes}}}
    del S, cidx, tok, slot, sc

    # acceptance of the best path vs the greedy walk through the T=0 verify, on
    # planted pair scores (a true slot path with +3 sigma on its transitions) and
    # a target whose arg-max is the true token at every position
    Bc, Vc = 2048, 4096
    S, pci, _, true_tok = synth.planted_path(23, Bc, L, Vc, mu=3.0)
    dS, dci = to_dev(torch, S, dev), to_dev(torch, pci, dev)
    dtg = to_dev(torch, synth.target_planted(24, true_tok, Vc, agree=1.0), dev)
    gtok, gslot, gq = api.walk(h, dS, dci, temperature=0.0)
    vtok, vslot, _ = api.walk_viterbi(h, dS, dci, want_score=False)
    ag, _ = api.verify(h, dtg, gtok, gslot, gq, dci, temperature=0.0)
    av, _ = api.verify(h, dtg, vtok, vslot, gq, dci, temperature=0.0)
    walk_ms = _timed(torch, lambda: api.walk(h, dS, dci, temperature=0.0, draft_tok=gtok, draft_slot=gslot,
                                             want_q=False))
    vit_ms = _timed(torch, lambda: api.walk_viterbi(h, dS, dci, draft_tok=vtok, draft_slot=vslot,
                                                    want_score=False))
    out["viterbi_vs_greedy"] = {"workload": f"B={Bc} L={L} V={Vc}, planted path mu=3 sigma=1",
                                "mean_accept_greedy": round(float(ag.double().mean()), 4),
                                "mean_accept_best_path": round(float(av.double().mean()), 4),
                                "greedy_walk_us": round(walk_ms * 1e3, 2), "best_path_us": round(vit_ms * 1e3, 2)}
    del dS, dci, dtg

    # projection-form selector: A, B projected from a shared [V, d] embedding for
    # the step's own candidates and gate (L2 flushed before each call)
    E = torch.randn((V, D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    WA = (torch.randn((R, D), generator=g, device=dev, dtype=torch.float32) / D ** 0.5).to(torch.bfloat16)
    WB = (torch.randn((R, D), generator=g, device=dev, dtype=torch.float32) / D ** 0.5).to(torch.bfloat16)
    P = torch.empty((nb * L * K + nb, 2 * R), dtype=torch.float32, device=dev)
    Sp = torch.empty((nb, L, K, K), dtype=torch.float32, device=dev)
    cv = cyc.vals.view(nb, L, K)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    ms_p = _timed(torch, lambda: (flush.zero_(), api.pair_scores_proj(h, ci, cv, cyc.lv, cyc.gate, E, WA, WB, P=P,
                                                                      S=Sp)), reps=9)
    ms_f = _timed(torch, lambda: flush.zero_(), reps=9)
    ms_p = max(ms_p - ms_f, 1e-6)
    del flush, E
    flops = (nb * L * K + nb) * 2 * R * D * 2.0
    tf = flops / (ms_p * 1e-3) / 1e12
    out["projection_selector"] = {
        "workload": f"B={nb} L={L} V={V} d={D}: projections of {nb * L * K + nb} tokens + pair scores",
        "ms": round(ms_p, 4), "table_form_pairs_ms_in_step": None,
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(tf / pk["bf16_tflops"], 4),
                     "note": "whole call (projection GEMM + pair kernel) against the projection's flops",
                     "traffic": profiled_traffic(["proj_kernel_B128_d5120.md"])}}
    del P, Sp, WA, WB

    # the conv fused into its producing GEMM (an output projection K = d) against the
    # library GEMM (cuBLAS, bf16 x) followed by the conv kernel; L2 flushed before each call
    Kp = D
    A = torch.randn((nb, L, Kp), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    Wp = (torch.randn((D, Kp), generator=g, device=dev, dtype=torch.float32) / Kp ** 0.5).to(torch.bfloat16)
    hs = torch.randn((nb, L, D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    x_prev, k0, k1, W_c = cyc.conv[0][1], cyc.conv[0][2], cyc.conv[0][3], cyc.conv[0][4]
    c_work = torch.empty(((api.gemm_conv2tap_workspace(h, nb, L, D) + 3) // 4,), dtype=torch.float32, device=dev)
    y = torch.empty((nb, L, D), dtype=torch.bfloat16, device=dev)
    x = torch.empty((nb * L, D), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    ms_f = _timed(torch, lambda: flush.zero_(), reps=9)
    fused = _timed(torch, lambda: (flush.zero_(), api.gemm_conv2tap(h, A, Wp, x_prev, hs, k0, k1, W_c, c_work=c_work,
                                                                    y=y)), reps=9) - ms_f
    unfused = _timed(torch, lambda: (flush.zero_(), torch.matmul(A.view(nb * L, Kp), Wp.t(), out=x),
                                     api.conv2tap(h, x.view(nb, L, D), x_prev, k0, k1, W_c, hs=hs, y=y)),
                     reps=9) - ms_f
    del flush
    flops = 2.0 * nb * L * D * (Kp + 2 * (D // 16))
    tf = flops / (fused * 1e-3) / 1e12
    out["conv_fused_gemm"] = {
        "workload": f"B={nb} L={L} K={Kp} d={D}: y = conv(A W^T), correction from a given hidden state",
        "fused_ms": round(fused, 4), "unfused_cublas_plus_conv_ms": round(unfused, 4),
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(tf / pk["bf16_tflops"], 4),
                     "note": "whole call (one persistent kernel: correction and fused tiles) against both GEMMs' flops",
                     "traffic": profiled_traffic(["gemm_conv_kernel_B128_K5120_d5120.md"])}}
    del A, Wp, hs, c_work, y, x

    r1, r16 = table1_recalls()
    Le = len(r1)
    gt = torch.randint(0, 1 << 20, (B_eval, Le), generator=g, device=dev, dtype=torch.int32)
    cand = torch.randint(1 << 21, 1 << 22, (B_eval, Le, K), generator=g, device=dev, dtype=torch.int32)
    u = torch.rand((B_eval, Le), generator=g, device=dev)
    top = u < torch.tensor(r1, device=dev)
    inside = (~top) & (u < torch.tensor(r16, device=dev))
    pos = torch.randint(1, K, (B_eval, Le, 1), generator=g, device=dev)
    cand[:, :, 0] = torch.where(top, gt, cand[:, :, 0])
    cand.scatter_(2, pos, torch.where(inside, gt, cand.gather(2, pos).squeeze(2)).unsqueeze(2))
    del u, top, inside, pos
    a1 = torch.empty((B_eval,), dtype=torch.int32, device=dev)
    a16 = torch.empty((B_eval,), dtype=torch.int32, device=dev)
    counts = torch.empty((Le, 4), dtype=torch.int64, device=dev)
    ms = _timed(torch, lambda: api.selector_eval(h, gt, cand, accept1=a1, accept16=a16, counts=counts))
    nbytes = B_eval * Le * (K * 4 + 4) + B_eval * 8 + Le * 4 * 8
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["selector_eval"] = {"workload": f"B={B_eval} L={Le}, Table 1 recalls planted", "ms": round(ms, 4),
                            "sequences_per_s": round(B_eval / (ms * 1e-3), 1),
                            "mean_accept_top1": round(float(a1.double().mean()), 4),
                            "mean_accept_top16_oracle": round(float(a16.double().mean()), 4),
                            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                                         "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                                         "traffic": _scaled_traffic("selector_eval_B524288.md", B_eval / 524288),
                                         "alg_bytes_per_launch": nbytes}}
    del gt, cand, a1, a16, counts
    return out


def run_e2e(torch, api, h, w, cyc, dev, args):
    """Same cycle through the public API from pinned host buffers: H2D of the
    step's inputs (activations, drafter logits, target logits, last verified
    tokens) and D2H of the acceptance lengths and emitted tokens, timed.  The
    inputs are double-buffered on the device: a copy stream brings in step i+1's
    inputs while step i computes (the host link, ~210 GB/s, is the bound)."""
    host = {
        "U": torch.from_numpy(w["U"][: B * L].view(np.int16)).pin_memory(),
        "target": cyc.target.view(torch.int16).cpu().pin_memory(),
        "lv": torch.from_numpy(w["last_verified"]).pin_memory(),
    }
    for a, (x, xp, *_rest) in enumerate(w["conv"]):
        host[f"x{a}"] = torch.from_numpy(x.view(np.int16)).pin_memory()
        host[f"xp{a}"] = torch.from_numpy(xp.view(np.int16)).pin_memory()
    res = {"acc": [torch.empty((B,), dtype=torch.int32).pin_memory() for _ in range(2)],
           "out": [torch.empty((B, L + 1), dtype=torch.int32).pin_memory() for _ in range(2)]}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for v in res.values() for t in v)
    # two device copies of the inputs: the cycle's own buffers and a second set
    sets = [{"U": cyc.U, "target": cyc.target, "lv": cyc.lv, "conv": cyc.conv},
            {"U": torch.empty_like(cyc.U), "target": torch.empty_like(cyc.target), "lv": torch.empty_like(cyc.lv),
             "conv": [tuple(torch.empty_like(t) if j < 2 else t for j, t in enumerate(c)) for c in cyc.conv]}]

    def dst_of(sset):
        d = {"U": sset["U"].view(torch.int16), "target": sset["target"].view(torch.int16), "lv": sset["lv"]}
        for a, (x, xp, *_rest) in enumerate(sset["conv"]):
            d[f"x{a}"] = x.view(torch.int16)
            d[f"xp{a}"] = xp.view(torch.int16)
        return d
    dsts = [dst_of(x) for x in sets]
    compute = torch.cuda.current_stream()
    copier = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    for e in free:
        e.record(compute)

    def copy_in(i):
        k = i % 2
        copier.wait_event(free[k])            # the step that last read this set is done
        with torch.cuda.stream(copier):
            for name in host:
                dsts[k][name].copy_(host[name], non_blocking=True)
        ready[k].record(copier)

    def compute_step(i):
        k = i % 2
        compute.wait_event(ready[k])
        cyc.U, cyc.target, cyc.lv, cyc.conv = sets[k]["U"], sets[k]["target"], sets[k]["lv"], sets[k]["conv"]
        cyc.step(seed_offset=2000 + i)
        free[k].record(compute)
        for j in range(2):
            res["acc"][j].copy_(cyc.acc[j], non_blocking=True)
            res["out"][j].copy_(cyc.out[j], non_blocking=True)

    def run(n, start):
        copy_in(start)
        for i in range(start, start + n):
            if i + 1 < start + n:
                copy_in(i + 1)
            compute_step(i)

    run(2, 0)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, args.steps // 2)
    t0.record()
    run(n, 2)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    # the cycle's buffers are left as they were
    cyc.U, cyc.target, cyc.lv, cyc.conv = sets[0]["U"], sets[0]["target"], sets[0]["lv"], sets[0]["conv"]
    return {"value": round(B * n / (ms * 1e-3), 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n, "ms_per_step": round(ms / n, 4),
            "overlap": "inputs double-buffered; copies of step i+1 overlap step i"}


def oracle_cycle(w, target_bits, nb, nthreads):
    """The oracle's own chain on the first nb sequences of the workload."""
    import oracle
    for x, xp, k0, k1, W in w["conv"]:
        cur = synth.bf16_bits(oracle.conv2tap(x[:nb], xp[:nb], k0, k1, W, nthreads=nthreads).astype(np.float32))
    ov, oi = oracle.topk(w["U"][: nb * L], nthreads=nthreads)
    ci, cv = oi.reshape(nb, L, K), ov.reshape(nb, L, K)
    H = oracle.gate(cur.reshape(nb * L, D), w["W_H"], None, nthreads=nthreads).reshape(nb, L, R)
    S, _ = oracle.pair_scores(ci, cv, w["last_verified"][:nb], H, w["A"], w["Bt"], nthreads=nthreads)
    S32 = S.astype(np.float32)
    accs = []
    for T in (0.0, 1.0):
        tok, slot, q, _ = oracle.walk(S32, ci, temperature=T, seed=1, nthreads=nthreads)
        acc, _, _ = oracle.verify(target_bits[:nb], tok, slot, q, ci, temperature=T, seed=1, nthreads=nthreads)
        accs.append(acc)
    return accs


def cpu_info():
    """CPU model (lscpu, else /proc/cpuinfo), logical CPUs and the CPUs this process may use."""
    model = None
    try:
        txt = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in txt.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    model = ln.split(":", 1)[1].strip()
                    break
    return {"model": model, "logical_cpus": os.cpu_count(), "usable_cpus": len(os.sched_getaffinity(0))}


def _repeat(fn, repeats):
    ts = []
    for _ in range(repeats):
        t = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t)
    return ts


def run_cpu_baseline(w, target_bits, sample_all=64, sample_one=4, repeats=3, lm_rows_all=64, lm_rows_one=2):
    """The oracle as it stands on the host cores: the full cycle on a sample of the
    workload's sequences, all cores and one thread, several repeats each; and the
    LM head + top-16 oracle's time per row on the C4 shapes (d=5120, V=151936)."""
    import oracle
    threads = oracle.default_threads()
    used = oracle.threads_used(threads)
    t_all = _repeat(lambda: oracle_cycle(w, target_bits, sample_all, threads), repeats)
    t_one = _repeat(lambda: oracle_cycle(w, target_bits, sample_one, 1), repeats)
    med_all, med_one = statistics.median(t_all), statistics.median(t_one)
    # C4: W is a seeded N(0, 0.02^2) block of 4096 rows tiled to V rows (drawing all
    # 778M values would take longer than the timing; the oracle's cost does not
    # depend on the values)
    block = synth.normal_bits(4, (4096, D), std=0.02)
    W = np.tile(block, (-(-V // 4096), 1))[:V]
    hidden = synth.normal_bits(5, (lm_rows_all, D))
    lm_all = _repeat(lambda: oracle.lmhead_topk(hidden, W, np.arange(lm_rows_all), nthreads=threads), repeats)
    lm_one = _repeat(lambda: oracle.lmhead_topk(hidden, W, np.arange(lm_rows_one), nthreads=1), repeats)
    del W
    return {"value": round(sample_all / med_all, 4), "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"first {sample_all} of {B} sequences of the workload, one full cycle, median of "
                      f"{repeats} repeats on {used} threads",
            "cpu": cpu_info(),
            "all_cores": {"threads": used, "sequences": sample_all, "seconds": [round(t, 3) for t in t_all],
                          "blocks_per_s": round(sample_all / med_all, 4)},
            "single_thread": {"threads": 1, "sequences": sample_one, "seconds": [round(t, 3) for t in t_one],
                              "blocks_per_s": round(sample_one / med_one, 4)},
            "lmhead_topk_per_row": {
                "workload": f"fused LM-head top-16 rows, d={D} V={V} (fp64 dot products)",
                "all_cores_s_per_row": round(statistics.median(lm_all) / lm_rows_all, 4),
                "all_cores_rows": lm_rows_all,
                "single_thread_s_per_row": round(statistics.median(lm_one) / lm_rows_one, 4),
                "single_thread_rows": lm_rows_one, "repeats": repeats,
                "M1024_extrapolated_s_all_cores": round(1024 * statistics.median(lm_all) / lm_rows_all, 1)}}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one full cycle over a
    bounded sample of the workload's sequences, on all host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    sample = 4
    w = make_host_workload(sample)
    rng_tok = np.random.default_rng(7).integers(0, V, (sample, L)).astype(np.int32)
    target = synth.target_planted(7, rng_tok, V, agree=0.85, plant=8.0)
    threads = oracle.default_threads()
    used = oracle.threads_used(threads)
    for _ in range(args.warmup):
        oracle_cycle(w, target, sample, threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_cycle(w, target, sample, threads)
    dt = time.perf_counter() - t
    value = sample * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": WORKLOAD, "B": B, "L": L, "V": V, "d": D,
                       "sample_sequences_per_step": sample,
                       "target": "planted (0.85 agreement) on seeded random tokens, not on the oracle's own "
                                 "draft, so acceptance lengths differ from the GPU arm's; the cost per cycle "
                                 "is that of the same stages at the same shapes"},
            "cpu": cpu_info(),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": f"{sample} of {B} sequences per step, full cycle"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dflash2", choices=["dflash2", "reference"])
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-lmhead", dest="lmhead", action="store_false")
    ap.add_argument("--no-next", dest="next", action="store_false")
    ap.add_argument("--no-small", dest="small", action="store_false")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
