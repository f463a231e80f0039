"""Benchmark of the self-speculative decode round on one GB300 (or N replicas).

Default workload: text-region decode on the 0.5B-class bf16 decoder (16 layers,
hidden 1536, 12 q / 4 kv heads of 128, SwiGLU 4096, vocab 65536), random-init
N(0, 0.02) weights, a 1024-row N(0, 1) synthetic prefix, B = 32, 73 output
tokens, batch 1, natural drafts.  One step = one decode of that region
through the C ABI (the whole round loop on the device); the prefill that sets
up each step is not timed (decode-only, the pages' Table 3 definition).

Prints one JSON line.  `--impl reference` times the CPU oracle instead.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from self_speculative_block_gb300 import synth  # noqa: E402

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0


def peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.th = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# --------------------------------------------------------------------------- workload

def workload(name: str):
    return synth.WORKLOADS[name]


def round_bytes(cfg: synth.ModelConfig, p: int, B: int) -> int:
    """Algorithmic HBM bytes of one round: all weights twice (draft + verify),
    the KV cache read by each forward, and the 2 (B + 1) KV rows written."""
    kv_tok = cfg.kv_bytes_per_token()
    return (2 * cfg.weight_bytes_per_forward() + (p + B + 1) * kv_tok + (p + B + 2) * kv_tok
            + 2 * (B + 1) * kv_tok)


def kernels_per_forward(cfg: synth.ModelConfig) -> int:
    # embed + per layer (qkv, attention, o, gate/up, down) + LM head; RMSNorm is folded into the GEMMs
    return 1 + 5 * cfg.n_layers + 1


def kernels_per_round(cfg: synth.ModelConfig) -> int:
    # plan, draft forward, override, plan, verify forward, accept
    return 2 * kernels_per_forward(cfg) + 4


# --------------------------------------------------------------------------- CPU oracle arm

class OracleArm:
    """The CPU oracle on a bounded sample of the workload: one untimed prefill,
    then each sample runs self-speculative rounds from a copy of that state
    until ~`seconds` of round time or the end of the workload.

    The 16-request page batch is sampled on its first request (the oracle
    decodes requests one after another, so its rate is per request).  Forced
    workloads first decode, untimed, an AR-greedy continuation of at most
    `ref_seconds` of oracle time; the forced drafts copy it, and a sample stops
    where it runs out."""

    def __init__(self, wl, ref_seconds: float = 20.0):
        import oracle
        self.oracle = oracle
        self.wl = wl
        cfg = wl.model
        if wl.n_requests > 1:
            prefix_lens, new_lens = synth.batch_lengths(wl.n_requests)
            self.P, self.max_new, seed = prefix_lens[0], new_lens[0], synth.REQUEST_PREFIX_SEED0
        else:
            self.P, self.max_new, seed = wl.prefix_len, wl.max_new, synth.PREFIX_SEED
        W = synth.make_weights(cfg)
        self.model = oracle.Model(W, cfg)
        del W
        prefix = synth.make_prefix(cfg, self.P, seed=seed).astype(np.float64)
        self.st0 = oracle.prefill(self.model, prefix)
        self.ref, self.override = None, None
        if wl.forced_mean is not None:
            st = self._copy()
            t0 = time.perf_counter()
            while len(st.out) < self.max_new and time.perf_counter() - t0 < ref_seconds:
                oracle.ar_step(self.model, st)
            self.ref = list(st.out)
            sched = synth.accept_schedule(wl.forced_mean, self.max_new, seed=synth.SCHEDULE_SEED)
            self.override = oracle.forced_override(self.ref, sched, cfg.vocab)

    def _copy(self):
        s = self.st0
        return self.oracle.State(list(s.cache_k), list(s.cache_v), s.x0, list(s.out))

    def sample(self, seconds: float):
        o, wl = self.oracle, self.wl
        st = self._copy()
        committed, rounds, t_total = 0, 0, 0.0
        while len(st.out) < self.max_new and t_total < seconds:
            if self.ref is not None and len(self.ref) < self.max_new and len(st.out) + wl.block + 2 > len(self.ref):
                break
            t0 = time.perf_counter()
            log = o.selfspec_round(self.model, st, wl.block, self.max_new, override=self.override,
                                   round_index=rounds)
            t_total += time.perf_counter() - t0
            committed += len(log.committed)
            rounds += 1
        try:
            from threadpoolctl import threadpool_info
            cores = max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count() or 1])
        except Exception:
            cores = os.cpu_count() or 1
        what = "natural drafts" if self.ref is None else f"forced drafts, geometric mean {wl.forced_mean}"
        req = f"request 0 ({self.P}-row prefix) of " if wl.n_requests > 1 else f"{self.P}-row prefill of "
        return {"value": committed / max(t_total, 1e-9), "unit": "tokens/s", "cores": int(cores), "kind": "oracle",
                "sample": f"{rounds} self-speculative rounds (B={wl.block}, fp64 NumPy, {what}) after an untimed "
                          f"{req}{wl.name}; {committed} tokens in {t_total:.1f} s"}


# --------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gocr", choices=["gocr", "reference"])
    ap.add_argument("--workload", default="text", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = workload(args.workload)
    metric = "committed tokens/s per region at B=32 (batch 1)"

    if args.impl == "reference":
        if rank != 0:
            return
        vals, secs, samples = [], [], []
        arm = OracleArm(wl)
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            s = arm.sample(seconds=max(2.0, args.cpu_seconds / max(1, args.steps)))
            if i >= args.warmup:
                vals.append(s["value"])
                secs.append(time.perf_counter() - t0)
                samples.append(s)
        v = statistics.median(vals)
        cb = dict(samples[-1])
        cb["value"] = v
        config = {"workload": wl.name, "prefix": arm.P, "B": wl.block, "max_new": arm.max_new,
                  "batch": 1, "parallelism": "host cores",
                  "drafts": "natural" if wl.forced_mean is None else f"forced, geometric mean {wl.forced_mean}"}
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": cb, "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                            "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    from self_speculative_block_gb300 import gocr

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    cfg = wl.model
    W = synth.make_weights(cfg)
    hbm, peak_kind = peaks()
    B = wl.block
    kind = args.workload
    if kind == "batch":
        prefix_lens, new_lens = synth.batch_lengths(wl.n_requests)
        max_ctx = max(prefix_lens) + max(new_lens) + B + 8
        n_req = wl.n_requests
    elif kind == "sweep":
        max_ctx = wl.prefix_len + wl.max_new + max(synth.SWEEP_BLOCKS) + 8
        prefix_lens, new_lens, n_req = [wl.prefix_len], [wl.max_new], 1
    else:
        max_ctx = wl.prefix_len + wl.max_new + B + 8
        prefix_lens, new_lens, n_req = [wl.prefix_len], [wl.max_new], 1
    dec = gocr.Decoder(cfg, W, max_ctx=max_ctx, max_block=max(B, max(synth.SWEEP_BLOCKS) if kind == "sweep" else B),
                       max_requests=n_req, device=str(dev))
    prefixes = []
    for r in range(n_req):
        seed = synth.REQUEST_PREFIX_SEED0 + r if kind == "batch" else synth.PREFIX_SEED
        pb = synth.make_prefix(cfg, prefix_lens[r], seed=seed)
        bits = np.ascontiguousarray(synth.bf16_bits(pb) if cfg.dtype == synth.BF16 else pb)
        prefixes.append((bits, torch.from_numpy(bits.view(np.int16) if cfg.dtype == synth.BF16 else bits).to(dev)))
    refs = []
    if wl.forced_mean is not None:
        # the AR-greedy continuation each forced draft copies (setup, not timed)
        for r in range(n_req):
            dec.prefill(r, prefixes[r][1])
            ref, _ = dec.decode(r, gocr.MODE_AR, 0, new_lens[r])
            refs.append(ref)

    def arm(mean, seed_off=0):
        for r in range(n_req):
            dec.set_draft_override(r, refs[r], synth.accept_schedule(mean, new_lens[r], seed=synth.SCHEDULE_SEED + r + seed_off))

    def step(Bv=B):
        for r in range(n_req):
            dec.prefill(r, prefixes[r][1])
        if n_req == 1:
            out, st = dec.decode(0, gocr.MODE_SELFSPEC, Bv, new_lens[0])
            return st["device_ms"], st["committed"], st["rounds"]
        outs, sts = dec.decode_batch(list(range(n_req)), gocr.MODE_SELFSPEC, Bv, new_lens)
        return sts[0]["device_ms"], sum(x["committed"] for x in sts), max(x["rounds"] for x in sts)

    sweep = None
    if kind == "sweep":
        sweep = []
        for Bv in synth.SWEEP_BLOCKS:
            for mean in synth.SWEEP_MEANS:
                arm(mean)
                for _ in range(2):
                    step(Bv)
                ms_l, tok_l, rd_l = [], 0, 0
                for _ in range(3):
                    ms, tk, rd = step(Bv)
                    ms_l.append(ms); tok_l += tk; rd_l += rd
                sweep.append({"B": Bv, "mean_accepted": mean, "round_us": 1e3 * sum(ms_l) / rd_l,
                              "tokens_per_s": tok_l / (sum(ms_l) / 1e3), "tpf": tok_l / (2 * rd_l)})
    if wl.forced_mean is not None:
        arm(wl.forced_mean)

    for _ in range(args.warmup):
        step()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    dev_ms, tokens, rounds = [], 0, 0
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            ms, tk, rd = step()
            dev_ms.append(ms)
            tokens += tk
            rounds += rd
    torch.cuda.synchronize()
    total_s = sum(dev_ms) / 1e3
    if world > 1:
        total_s, tokens = replica_totals(total_s, tokens, dev)
    value = tokens / total_s
    ms_per_step = sum(dev_ms) / len(dev_ms)
    round_us = 1e3 * sum(dev_ms) / rounds
    # round roofline: algorithmic bytes of an average round at the mean cache length
    p_mid = int(np.mean(prefix_lens) + np.mean(new_lens) / 2)
    rb = round_bytes(cfg, p_mid, B)
    if n_req > 1:  # weights once per forward, every request's KV
        rb = 2 * cfg.weight_bytes_per_forward() + n_req * (round_bytes(cfg, p_mid, B) - 2 * cfg.weight_bytes_per_forward())
    round_frac = (rb / (hbm * 1e9)) / (round_us * 1e-6)

    # dominant kernel: the split-K GEMM on one forward's weight matrices, timed live
    kern = kernel_roofline(cfg, B, hbm, dev)

    # end to end through the C ABI with host buffers: H2D prefixes, prefill, decode, D2H tokens
    pinned = [torch.from_numpy(b.view(np.int16) if cfg.dtype == synth.BF16 else b).pin_memory() for b, _ in prefixes]
    e2e_tok, e2e_s = 0, 0.0
    for _ in range(max(1, args.steps)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for r in range(n_req):
            dec.prefill(r, pinned[r])
        if n_req == 1:
            out, st = dec.decode(0, gocr.MODE_SELFSPEC, B, new_lens[0])
            e2e_tok += st["committed"]
        else:
            outs, sts = dec.decode_batch(list(range(n_req)), gocr.MODE_SELFSPEC, B, new_lens)
            e2e_tok += sum(x["committed"] for x in sts)
        e2e_s += time.perf_counter() - t0
    h2d = int(sum(b.nbytes for b, _ in prefixes))
    d2h = int(sum(new_lens) * 4)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dec.close()
        del W
        torch.cuda.empty_cache()
        cpu = OracleArm(wl).sample(seconds=args.cpu_seconds)
    launches = rounds * kernels_per_round(cfg) + args.steps  # + one begin-decode kernel per call
    if rank == 0:
        config = {"workload": wl.name, "prefix": prefix_lens if n_req > 1 else prefix_lens[0], "B": B,
                  "max_new": new_lens if n_req > 1 else new_lens[0], "batch": n_req,
                  "parallelism": "replicas" if world > 1 else "single-gpu",
                  "l2": "inputs larger than L2 (1.0 GB of weights per forward)",
                  "drafts": "natural" if wl.forced_mean is None else f"forced, geometric mean {wl.forced_mean}"}
        line = {
            "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if cfg.dtype == synth.BF16 else "f32", "data": "synthetic",
            "config": config,
            "round_us": round_us, "rounds_per_step": rounds / args.steps,
            "tpf": tokens / (2 * rounds),
            "round_roofline": {"bytes": rb, "peak_gbs": hbm, "frac": round_frac, "peak": peak_kind},
            "roofline": kern,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_tok / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clk.summary(),
        }
        if sweep is not None:
            line["sweep"] = sweep
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


GEMM_SOURCES = ("gemm_tc.cu", "gemm.cu", "epilogue.cuh", "tc.cuh", "kernels.cuh", "common.cuh")
GEMM_PROFILE = os.path.join(ROOT, "profiles", "gemm_tc_decode_sweep.md")


def replica_totals(total_s: float, tokens: int, device) -> tuple[float, int]:
    """N replicas (one process per GPU, an initialised process group): the
    slowest rank's timed seconds and the tokens all ranks committed, so that
    the whole-job rate is tokens / seconds."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(total_s), float(tokens)], dtype=torch.float64, device=device)
    tt = [torch.zeros_like(t) for _ in range(dist.get_world_size())]
    dist.all_gather(tt, t)
    return max(float(x[0]) for x in tt), sum(int(round(float(x[1]))) for x in tt)


def gemm_sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "self_speculative_block_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the GEMM sweep from the committed ncu summary,
    or None when the kernel sources changed since that capture."""
    try:
        kv = dict(line.split(":", 1) for line in open(GEMM_PROFILE).read().splitlines()
                  if line.startswith(("traffic_bytes_per_launch:", "gemm_sources_digest:")))
    except (OSError, ValueError):
        return None
    if kv.get("gemm_sources_digest", "").strip() != gemm_sources_digest():
        return None
    return float(kv["traffic_bytes_per_launch"])


def kernel_roofline(cfg, B, hbm, dev):
    """The split-K GEMM kernel on one forward's 65 weight launches (every
    layer's packed QKV, O, packed gate/up and down, then the LM head) at the
    decode launch shape: B + 1 tokens as bf16 hi and lo planes, each launch
    with programmatic dependent launch, as the forward launches them (the
    forward's fused epilogues are a plain fp32 store here).  Timed with CUDA
    events on the stream it is launched on; the matrices total ~1 GB, more
    than L2, so every launch streams its weights from HBM."""
    import torch
    from self_speculative_block_gb300.profile_cases import GemmSweep
    sw = GemmSweep(cfg, B + 1, dev)
    g = sw.graph()
    g.replay()
    s = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(reps):
        g.replay()
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * len(sw.shapes))
    alg = sw.algorithmic_bytes()
    ach = alg / (ms * 1e-3) / 1e9
    n = len(sw.shapes)
    del sw
    return {"kernel": f"gemm_tc_kernel (tcgen05 split-K GEMM), one forward's {n} weight launches",
            "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
            "traffic": profiled_traffic(), "launch_us": ms * 1e3, "algorithmic_bytes": alg,
            "tokens": B + 1, "planes": 2, "launches": n}


if __name__ == "__main__":
    main()
