"""Benchmark of the self-speculative decode round on one GB300 (or N replicas).

Default workload: text-region decode on the 0.5B-class bf16 decoder (16 layers,
hidden 1536, 12 q / 4 kv heads of 128, SwiGLU 4096, vocab 65536), random-init
N(0, 0.02) weights, a 1024-row N(0, 1) synthetic prefix, B = 32, 73 output
tokens, batch 1, natural drafts.  One step = one decode of that region
through the C ABI (the whole round loop on the device); the prefill that sets
up each step is not timed (decode-only, the pages' Table 3 definition).

Prints one JSON line.  Besides the workload's own numbers it carries, for
the default workload: the AR-greedy decode of the same region (the method's
speed-up is self-speculative over AR), the table region with forced
acceptance, the GEMMs' roofline as the forward runs them and as a kernel
alone, the pages' equality protocol against the fp64 oracle, and the fp32
oracle's rate on all host cores and on one.  `--impl reference` times the
CPU oracle instead.
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
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor TFLOP/s (burst) and its source."""
    try:
        with open(MEASURED_PEAKS) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


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
    """embed + per layer (QKV, attention partial, attention merge, O, gate/up,
    down; fp32 models: one attention kernel) + LM head; RMSNorm is folded into
    the GEMMs."""
    att = 2 if cfg.dtype == synth.BF16 else 1
    return 1 + (4 + att) * cfg.n_layers + 1


def kernels_per_round(cfg: synth.ModelConfig) -> int:
    # plan, draft forward, override, plan, verify forward, accept
    return 2 * kernels_per_forward(cfg) + 4


def kernels_per_ar_step(cfg: synth.ModelConfig) -> int:
    # plan, forward, commit
    return kernels_per_forward(cfg) + 2


# --------------------------------------------------------------------------- CPU oracle leg

BLAS_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def blas_threads() -> int:
    """Threads NumPy's BLAS runs with: the thread variables when set (they
    take effect when NumPy loads), else one per host core (the default)."""
    for v in BLAS_THREAD_VARS:
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count() or 1


def cpu_sample_subprocess(workload_name: str, seconds: float, threads: int) -> dict:
    """One oracle sample in a fresh interpreter whose BLAS runs `threads`
    threads (fixed by the thread variables before NumPy loads)."""
    env = dict(os.environ)
    for v in BLAS_THREAD_VARS:
        env[v] = str(threads)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", "--workload", workload_name,
                        "--cpu-seconds", str(seconds)], env=env, capture_output=True, text=True, timeout=1800)
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not lines:
        return {"error": (r.stderr or r.stdout)[-400:]}
    return json.loads(lines[-1])


class OracleArm:
    """The CPU oracle on a bounded sample of a workload, in fp32 (the oracle's
    timing precision): one untimed prefill, then each sample runs
    self-speculative rounds from a copy of that state until ~`seconds` of
    round time or the end of the workload.

    The 16-request page batch is sampled on its first request (the oracle
    decodes requests one after another, so its rate is per request).  Forced
    workloads first decode, untimed, an AR-greedy continuation of at most
    `ref_seconds` of oracle time; the forced drafts copy it, and a sample stops
    where it runs out."""

    def __init__(self, wl, ref_seconds: float = 20.0, dtype=np.float32):
        import oracle
        self.oracle = oracle
        self.wl = wl
        self.dtype = dtype
        cfg = wl.model
        if wl.n_requests > 1:
            prefix_lens, new_lens = synth.batch_lengths(wl.n_requests)
            self.P, self.max_new, seed = prefix_lens[0], new_lens[0], synth.REQUEST_PREFIX_SEED0
        else:
            self.P, self.max_new, seed = wl.prefix_len, wl.max_new, synth.PREFIX_SEED
        W = synth.make_weights(cfg)
        self.model = oracle.Model(W, cfg, dtype=dtype)
        del W
        prefix = synth.make_prefix(cfg, self.P, seed=seed).astype(dtype)
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
        """Rounds for ~seconds, on the BLAS threads this process runs."""
        o, wl = self.oracle, self.wl
        st = self._copy()
        committed, rounds, t_total = 0, 0, 0.0
        cores = blas_threads()
        while len(st.out) < self.max_new and t_total < seconds:
            if self.ref is not None and len(self.ref) < self.max_new and len(st.out) + wl.block + 2 > len(self.ref):
                break
            t0 = time.perf_counter()
            log = o.selfspec_round(self.model, st, wl.block, self.max_new, override=self.override,
                                   round_index=rounds)
            t_total += time.perf_counter() - t0
            committed += len(log.committed)
            rounds += 1
        what = "natural drafts" if self.ref is None else f"forced drafts, geometric mean {wl.forced_mean}"
        req = f"request 0 ({self.P}-row prefix) of " if wl.n_requests > 1 else f"{self.P}-row prefill of "
        prec = "fp32" if self.dtype == np.float32 else "fp64"
        return {"value": committed / max(t_total, 1e-9), "unit": "tokens/s", "cores": int(cores), "kind": "oracle",
                "sample": f"{rounds} self-speculative rounds (B={wl.block}, {prec} NumPy, {what}) after an untimed "
                          f"{req}{wl.name}; {committed} tokens in {t_total:.1f} s"}


def equality_record(cfg, prefix, out, ar_out):
    """The pages' equality protocol (GravityOCR review, Appendix B.3) for one
    region: the GPU's committed tokens replayed in the fp64 oracle by one causal
    pass over [prefix, out[:-1]] (teacher forcing), the fraction of positions
    whose oracle argmax is the GPU's token, the first divergence and the
    oracle's top-two margin there, and whether the GPU's self-speculative
    output equals its own AR output."""
    import oracle
    W = synth.make_weights(cfg)
    model = oracle.Model(W, cfg)
    del W
    P = prefix.shape[0]
    toks = [int(t) for t in out]
    logits, _, _ = oracle.prefill_cache(model, prefix.astype(np.float64), toks[:-1])
    rows = logits[P - 1:P - 1 + len(toks)]
    am = np.argmax(rows, axis=-1)
    agree = am == np.asarray(toks)
    first = int(np.argmin(agree)) if not agree.all() else None
    margins = [oracle.top2_margin(r) for r in rows]
    rec = {"tokens": len(toks), "argmax_agreement": float(agree.mean()), "first_divergence": first,
           "median_top2_margin_nats": float(np.median(margins)),
           "selfspec_equals_gpu_ar": bool(list(out) == list(ar_out)),
           "oracle": "fp64 NumPy, one causal pass over the prefix and the GPU's tokens"}
    if first is not None:
        rec["top2_margin_at_first_divergence_nats"] = margins[first]
        rec["gpu_token_gap_at_first_divergence_nats"] = float(rows[first].max() - rows[first][toks[first]])
    return rec


# --------------------------------------------------------------------------- GPU timing

def time_decode(dec, prefixes, n_req, new_lens, B, mode, steps, warmup, clk=None):
    """warmup untimed, then `steps` timed decodes (each after an untimed
    prefill); device time from the library's CUDA events on its stream."""
    from self_speculative_block_gb300 import gocr

    def one():
        for r in range(n_req):
            dec.prefill(r, prefixes[r][1])
        if n_req == 1:
            out, st = dec.decode(0, mode, B, new_lens[0])
            return st["device_ms"], st["committed"], st["rounds"], st["forwards"], [out]
        outs, sts = dec.decode_batch(list(range(n_req)), mode, B, new_lens)
        return (sts[0]["device_ms"], sum(x["committed"] for x in sts), max(x["rounds"] for x in sts),
                max(x["forwards"] for x in sts), outs)

    for _ in range(warmup):
        one()
    import torch
    torch.cuda.synchronize()
    ms, tok, rd, fw, outs = [], 0, 0, 0, None
    ctx = clk if clk is not None else _Null()
    with ctx:
        for _ in range(steps):
            m, t, r, f, outs = one()
            ms.append(m)
            tok += t
            rd += r
            fw += f
    torch.cuda.synchronize()
    return {"ms": ms, "tokens": tok, "rounds": rd, "forwards": fw, "outs": outs}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def upload_prefixes(cfg, lens, seeds, dev):
    import torch
    res = []
    for n, seed in zip(lens, seeds):
        pb = synth.make_prefix(cfg, n, seed=seed)
        bits = np.ascontiguousarray(synth.bf16_bits(pb) if cfg.dtype == synth.BF16 else pb)
        res.append((bits, torch.from_numpy(bits.view(np.int16) if cfg.dtype == synth.BF16 else bits).to(dev), pb))
    return res


def table_record(cfg, W, hbm, dev, steps, warmup):
    """The table region (prefix 2048, 872 tokens, B = 32, forced acceptance of
    geometric mean 9): round time, rate, TPF, round roofline, and the AR
    decode of the same region (the continuation the forced drafts copy)."""
    from self_speculative_block_gb300 import gocr
    wl = synth.WORKLOADS["table"]
    B = wl.block
    dec = gocr.Decoder(cfg, W, max_ctx=wl.prefix_len + wl.max_new + B + 8, max_block=B, device=str(dev))
    try:
        prefixes = upload_prefixes(cfg, [wl.prefix_len], [synth.PREFIX_SEED], dev)
        dec.prefill(0, prefixes[0][1])
        dec.decode(0, gocr.MODE_AR, 0, wl.max_new)  # warm-up of the AR graph
        ar = time_decode(dec, prefixes, 1, [wl.max_new], 0, gocr.MODE_AR, max(1, min(steps, 2)), 0)
        ref = ar["outs"][0]
        dec.set_draft_override(0, ref, synth.accept_schedule(wl.forced_mean, wl.max_new, seed=synth.SCHEDULE_SEED))
        ss = time_decode(dec, prefixes, 1, [wl.max_new], B, gocr.MODE_SELFSPEC, steps, warmup)
        dec.clear_draft_override(0)
        same = list(ss["outs"][0]) == list(ref)
    finally:
        dec.close()
    round_us = 1e3 * sum(ss["ms"]) / ss["rounds"]
    p_mid = int(wl.prefix_len + wl.max_new / 2)
    frac = (round_bytes(cfg, p_mid, B) / (hbm * 1e9)) / (round_us * 1e-6)
    tps = ss["tokens"] / (sum(ss["ms"]) / 1e3)
    ar_tps = ar["tokens"] / (sum(ar["ms"]) / 1e3)
    return {"workload": wl.name, "round_us": round_us, "tokens_per_s": tps, "tpf": ss["tokens"] / ss["forwards"],
            "rounds_per_step": ss["rounds"] / steps, "round_roofline_frac": frac,
            "ar_tokens_per_s": ar_tps, "ar_us_per_token": 1e6 / ar_tps, "speedup_vs_ar": tps / ar_tps,
            "selfspec_equals_ar": same, "steps": steps, "warmup": warmup}


def next_rows_record(cfg, W, hbm, dev, steps, warmup):
    """The decoding modes beyond the greedy round on the text region (prefix 1024, B = 32, 73
    tokens): direct block-diffusion decoding (threshold 0.9), self-speculative
    rounds with refined drafts (at most 4 draft forwards, draft threshold 0.9),
    sampling (temperature 1) self-speculative against AR sampling, each as
    committed tokens/s, tokens per forward and us per forward (the forwards'
    share of the per-forward weight roofline); and the joint-training mask's
    attention (one kernel launch over prefix 1024 + 3 x 512 packed rows, block
    32) as us per launch and attention TFLOP/s over the mask's visible
    (row, key) pairs.  Synthetic random-init weights: the decodes' confidence
    and acceptance are those of an untrained model, so these time the
    mechanisms, not the method's quality."""
    import torch
    from self_speculative_block_gb300 import gocr
    wl = synth.WORKLOADS["text"]
    B, n = wl.block, wl.max_new
    dec = gocr.Decoder(cfg, W, max_ctx=wl.prefix_len + n + B + 8, max_block=B, device=str(dev))
    rec = {"workload": wl.name}
    try:
        prefix = upload_prefixes(cfg, [wl.prefix_len], [synth.PREFIX_SEED], dev)[0][1]

        def run(mode, blk, **kw):
            ms = tok = fw = 0
            for i in range(warmup + steps):
                dec.prefill(0, prefix)
                _, sts = dec.decode_ex([0], mode, blk, [n], **kw)
                if i >= warmup:
                    ms += sts[0]["device_ms"]; tok += sts[0]["committed"]; fw += sts[0]["forwards"]
            us_fw = 1e3 * ms / fw
            return {"tokens_per_s": tok / (ms / 1e3), "tokens_per_forward": tok / fw, "us_per_forward": us_fw,
                    "forward_roofline_frac": (cfg.weight_bytes_per_forward() / (hbm * 1e9)) / (us_fw * 1e-6)}

        rec["direct_diffusion"] = dict(run(gocr.MODE_DIFFUSION, B, tau=0.9), tau=0.9, B=B)
        rec["refined_drafts"] = dict(run(gocr.MODE_REFINED, B, tau=0.9, draft_steps=4), tau=0.9, draft_steps=4, B=B)
        rec["sampling_selfspec"] = dict(run(gocr.MODE_SELFSPEC, B, temperature=1.0, seed=1), temperature=1.0, B=B)
        rec["sampling_ar"] = dict(run(gocr.MODE_AR, 0, temperature=1.0, seed=1), temperature=1.0)
    finally:
        dec.close()
    # the joint-training mask as a second key interval per row
    from self_speculative_block_gb300.profile_cases import TrainMask
    tm = TrainMask(cfg, dev)
    for _ in range(3):
        tm.run()
    torch.cuda.synchronize()
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        tm.run()
    e1.record()
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / reps
    # tensor roofline: the hi/lo planes make 3 bf16 products for QK^T and 2 for
    # PV, 2.5 x the arithmetic of the visible pairs
    peak, peak_kind = bf16_peak()
    mma_tflops = 2.5 * tm.flops() / (us * 1e-6) / 1e12
    rec["training_mask_attention"] = {"rows": tm.L, "prefix": tm.P, "stream": tm.N, "block": tm.block,
                                      "us_per_launch": us, "visible_pairs": tm.visible_pairs(),
                                      "tflops": tm.flops() / (us * 1e-6) / 1e12,
                                      "roofline": {"bound": "tensor", "achieved": mma_tflops, "peak": peak,
                                                   "unit": "TFLOP/s", "frac": mma_tflops / peak,
                                                   "peak_kind": peak_kind,
                                                   "how": "bf16 MMA work of the visible pairs (hi/lo products) "
                                                          "over the call's CUDA-event time"}}
    return rec


# --------------------------------------------------------------------------- kernel rooflines

GEMM_SOURCES = ("gemm_tc.cu", "gemm.cu", "epilogue.cuh", "tc.cuh", "kernels.cuh", "common.cuh")
GEMM_TRAFFIC = os.path.join(ROOT, "profiles", "gemm_tc_decode_traffic.json")


def gemm_sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "self_speculative_block_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(key: str):
    """DRAM bytes per launch of a GEMM capture from the committed ncu summary
    (profiles/gemm_tc_decode_traffic.json), or None when the GEMM sources
    changed since that capture or it lacks the entry."""
    try:
        with open(GEMM_TRAFFIC) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(key)
    if not e or e.get("gemm_sources_digest") != gemm_sources_digest():
        return None
    return float(e["traffic_bytes_per_launch"])


def gemm_launch_bytes(cfg, T: int) -> float:
    """Mean algorithmic bytes of a forward's GEMM launch at T tokens: the
    weights, both bf16 input planes, and T x N fp32 of output."""
    from self_speculative_block_gb300.profile_cases import forward_gemm_shapes
    shapes = forward_gemm_shapes(cfg)
    return sum(n * k * 2 + 2 * T * k * 2 + T * n * 4 for n, k in shapes) / len(shapes)


def in_situ_gemm(cfg, W, wl, dev, hbm, round_us):
    """The GEMMs as the forward runs them (fused epilogues, programmatic
    dependent launch, inside a captured graph).  A handle with launch
    timelines (GOCR_OP_TRACE) runs the draft forward of the workload as a graph
    (GOCR_DEBUG_GRAPH); the timeline gives each launch's share of the forward
    (its end minus the previous launch's end).  The GEMMs' share of the
    CUDA-event round time of the timed decode, halved per forward, over the 65
    GEMM launches of a forward, is the in-situ time per launch."""
    from self_speculative_block_gb300 import gocr
    B = wl.block
    os.environ["GOCR_OP_TRACE"] = "1"
    try:
        dec = gocr.Decoder(cfg, W, max_ctx=wl.prefix_len + 2 * B + 16, max_block=B, device=str(dev))
    finally:
        del os.environ["GOCR_OP_TRACE"]
    try:
        dec.prefill(0, upload_prefixes(cfg, [wl.prefix_len], [synth.PREFIX_SEED], dev)[0][1])
        x0 = dec.state(0)[1]
        os.environ["GOCR_DEBUG_GRAPH"] = "1"
        try:
            shares = []
            for _ in range(5):
                dec.debug_forward(0, gocr.FWD_DRAFT, [x0] + [0] * B)
                tr = dec.read_kernel_trace().astype(np.int64)
                ends = tr[:, 3]
                chain = np.diff(np.concatenate([[tr[0, 0]], ends]))
                is_gemm = np.array([(i % 5) != 1 for i in range(tr.shape[0] - 1)] + [True])
                shares.append(float(chain[is_gemm].sum() / chain.sum()))
                run_us = float(np.mean((ends - tr[:, 1])[is_gemm]) / 1e3)
        finally:
            del os.environ["GOCR_DEBUG_GRAPH"]
    finally:
        dec.close()
    share = float(np.median(shares[1:]))
    n = int(is_gemm.sum())
    launch_us = round_us / 2 * share / n
    alg = gemm_launch_bytes(cfg, B + 1)
    ach = alg / (launch_us * 1e-6) / 1e9
    return {"kernel": "decode-forward GEMMs: gemm_tc_kernel (tcgen05 split-K, fused epilogues) and the LM head on gemm_tc_stream_kernel",
            "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
            "traffic": profiled_traffic("draft_forward"), "launch_us": launch_us, "algorithmic_bytes": alg,
            "gemm_share_of_forward": share, "launches_per_forward": n, "trace_run_us": run_us,
            "how": "round CUDA-event time / 2 x GEMM share of the forward timeline / GEMM launches"}


def kernel_sweep(cfg, B, hbm, dev):
    """The split-K GEMM alone on one forward's 65 weight launches at the decode
    launch shape (B + 1 tokens as bf16 hi and lo planes, programmatic dependent
    launch, a plain fp32-store epilogue), captured in one CUDA graph and timed
    with CUDA events on its stream; ~1 GB of weights, more than L2."""
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
    return {"kernel": f"gemm_tc_kernel alone, one forward's {n} weight launches, plain-store epilogue",
            "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
            "traffic": profiled_traffic("sweep"), "launch_us": ms * 1e3, "algorithmic_bytes": alg}


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


# --------------------------------------------------------------------------- main

def reference_arm(args, wl, metric, world, rank):
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
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config,
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gocr", choices=["gocr", "reference"])
    ap.add_argument("--workload", default="text", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the workload's own line: no table, AR, in-situ or sweep records")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-sample", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_sample:  # one oracle sample of the workload (the CPU leg's worker)
        print(json.dumps(OracleArm(workload(args.workload)).sample(seconds=args.cpu_seconds)), flush=True)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = workload(args.workload)
    metric = "committed tokens/s per region at B=32 (batch 1)"

    if args.impl == "reference":
        return reference_arm(args, wl, metric, world, rank)

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
    extras = not args.no_extras and world == 1
    if kind == "batch":
        prefix_lens, new_lens = synth.batch_lengths(wl.n_requests)
        max_ctx = max(prefix_lens) + max(new_lens) + B + 8
        n_req = wl.n_requests
    else:
        max_ctx = wl.prefix_len + wl.max_new + B + 8
        prefix_lens, new_lens, n_req = [wl.prefix_len], [wl.max_new], 1
    dec = gocr.Decoder(cfg, W, max_ctx=max_ctx, max_block=B, max_requests=n_req, device=str(dev))
    seeds = [synth.REQUEST_PREFIX_SEED0 + r if kind == "batch" else synth.PREFIX_SEED for r in range(n_req)]
    prefixes = upload_prefixes(cfg, prefix_lens, seeds, dev)

    def ar_refs(d):
        # the AR-greedy continuation each forced draft copies (setup, not timed)
        out = []
        for r in range(n_req):
            d.prefill(r, prefixes[r][1])
            ref, _ = d.decode(r, gocr.MODE_AR, 0, new_lens[r])
            out.append(ref)
        return out

    def arm(d, refs_d, mean, seed_off=0):
        for r in range(n_req):
            d.set_draft_override(r, refs_d[r], synth.accept_schedule(mean, new_lens[r], seed=synth.SCHEDULE_SEED + r + seed_off))

    refs = ar_refs(dec) if wl.forced_mean is not None else []
    sweep = None
    if kind == "sweep":
        # one handle per block size, as a deployment would size it: a handle's
        # attention ranks are fixed for its largest forward
        sweep = []
        for Bv in synth.SWEEP_BLOCKS:
            dv = dec if Bv == B else gocr.Decoder(cfg, W, max_ctx=wl.prefix_len + wl.max_new + Bv + 8, max_block=Bv,
                                                  max_requests=n_req, device=str(dev))
            try:
                refs_v = refs if dv is dec else ar_refs(dv)
                for mean in synth.SWEEP_MEANS:
                    arm(dv, refs_v, mean)
                    r = time_decode(dv, prefixes, n_req, new_lens, Bv, gocr.MODE_SELFSPEC, 3, 2)
                    sweep.append({"B": Bv, "mean_accepted": mean, "round_us": 1e3 * sum(r["ms"]) / r["rounds"],
                                  "tokens_per_s": r["tokens"] / (sum(r["ms"]) / 1e3),
                                  "tpf": r["tokens"] / r["forwards"], "attention_ranks": dv.attention_ranks()})
            finally:
                if dv is not dec:
                    dv.close()
    if wl.forced_mean is not None:
        arm(dec, refs, wl.forced_mean)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    main_r = time_decode(dec, prefixes, n_req, new_lens, B, gocr.MODE_SELFSPEC, args.steps, args.warmup, clk=clk)
    dev_ms, tokens, rounds = main_r["ms"], main_r["tokens"], main_r["rounds"]
    total_s = sum(dev_ms) / 1e3
    if world > 1:
        total_s, tokens = replica_totals(total_s, tokens, dev)
    value = tokens / total_s
    ms_per_step = sum(dev_ms) / len(dev_ms)
    round_us = 1e3 * sum(dev_ms) / main_r["rounds"]
    # round roofline: algorithmic bytes of an average round at the mean cache length
    p_mid = int(np.mean(prefix_lens) + np.mean(new_lens) / 2)
    rb = round_bytes(cfg, p_mid, B)
    if n_req > 1:  # weights once per forward, every request's KV
        rb = 2 * cfg.weight_bytes_per_forward() + n_req * (round_bytes(cfg, p_mid, B) - 2 * cfg.weight_bytes_per_forward())
    round_frac = (rb / (hbm * 1e9)) / (round_us * 1e-6)

    # AR greedy on the same workload and handle (the method's speed-up is self-spec over AR)
    ar_rec, ar_outs = None, None
    if extras and wl.forced_mean is None:
        ar = time_decode(dec, prefixes, n_req, new_lens, 0, gocr.MODE_AR, args.steps, args.warmup)
        ar_tps = ar["tokens"] / (sum(ar["ms"]) / 1e3)
        ar_outs = ar["outs"]
        ar_rec = {"tokens_per_s": ar_tps, "us_per_token": 1e6 / ar_tps,
                  "forward_roofline_frac": (cfg.weight_bytes_per_forward() / (hbm * 1e9)) / (1e-6 * 1e6 / ar_tps),
                  "speedup_of_selfspec": value / ar_tps,
                  "selfspec_equals_ar": [list(a) for a in ar_outs] == [list(o) for o in main_r["outs"]]}

    # end to end through the C ABI with host buffers: H2D prefixes, prefill, decode, D2H tokens
    pinned = [torch.from_numpy(b.view(np.int16) if cfg.dtype == synth.BF16 else b).pin_memory() for b, _, _ in prefixes]
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
    h2d = int(sum(b.nbytes for b, _, _ in prefixes))
    d2h = int(sum(new_lens) * 4)
    dec.close()

    # dominant kernel: the GEMMs in situ, and the GEMM alone on the forward's shapes
    kern, sweep_k, table = None, None, None
    if cfg.dtype == synth.BF16 and world == 1:
        kern = in_situ_gemm(cfg, W, wl if kind != "batch" else synth.WORKLOADS["text"], dev, hbm, round_us) \
            if kind != "batch" else None
        if extras:
            sweep_k = kernel_sweep(cfg, B, hbm, dev)
    nxt = None
    if extras and kind == "text":
        table = table_record(cfg, W, hbm, dev, args.steps, args.warmup)
        nxt = next_rows_record(cfg, W, hbm, dev, min(args.steps, 3), 1)

    cpu, equality = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del W
        torch.cuda.empty_cache()
        if extras and ar_outs is not None and n_req == 1:
            equality = equality_record(cfg, prefixes[0][2], main_r["outs"][0], ar_outs[0])
        # the fp32 oracle on every host core and on one, each in its own
        # interpreter so that its BLAS thread count is the one stated
        cpu = cpu_sample_subprocess(args.workload, args.cpu_seconds, os.cpu_count() or 1)
        one = cpu_sample_subprocess(args.workload, args.cpu_seconds / 2, 1)
        cpu["dtype"] = "f32"
        cpu["single_thread"] = {k: one.get(k) for k in ("value", "unit", "cores", "sample", "error") if k in one}
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
            "tpf": tokens / main_r["forwards"] if world == 1 else None,
            "round_roofline": {"bytes": rb, "peak_gbs": hbm, "frac": round_frac, "peak": peak_kind},
            "roofline": kern,
            "roofline_sweep": sweep_k,
            "ar": ar_rec,
            "table": table,
            "next": nxt,
            "equality": equality,
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


if __name__ == "__main__":
    main()
