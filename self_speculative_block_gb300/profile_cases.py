"""Small, self-contained launches of the hot kernels for capture under a profiler.

    python -m self_speculative_block_gb300.profile_cases draft [B]
        0.5B-class bf16 decoder, 1024-row synthetic prefill, then two draft
        forwards (B = 32 unless given: B + 1 rows).  The prefill (1024 rows)
        launches gemm_tc_seq_kernel 64 times, gemm_tc_kernel once (the LM
        head of its last row) and attention_part_kernel /
        attention_merge_kernel 16 times each; the draft forwards launch
        gemm_tc_kernel (65 per forward), so the first draft forward's QKV /
        O / gate-up / down GEMMs are launches 1..4 of `-k regex:gemm_tc_kernel`
        (65..68 of `-k regex:gemm_tc`, which also matches the prefill's
        kernel) and its first attention is attention_part and
        attention_merge launch 16.
    python -m self_speculative_block_gb300.profile_cases sweep
        The split-K GEMM over one forward's 65 weight matrices (16 x packed
        QKV, O, packed gate/up, down, then the LM head) at the decode launch
        shape: 33 tokens as bf16 hi and lo planes, launched with programmatic
        dependent launch as the forward launches them.  Runs the sweep once,
        then once more as a CUDA graph (gemm_tc launches 65..129 are the
        graph's).

    python -m self_speculative_block_gb300.profile_cases batch
        The 16-request page batch: 16 ragged prefills (each one plan, one
        embed, 65 GEMM, 16 attention partial, 16 attention merge and one
        finishing launch: 100 launches), then one batched self-speculative
        round (B = 32, 16 x 33 = 528 rows per forward).  Run it with
        GOCR_HOST_LOOP=1 so that the round's kernels are profilable: they
        start at launch 1600.

    python -m self_speculative_block_gb300.profile_cases train_mask
        The joint-training mask's attention over the packed sequence [prefix
        1024, clean 512, corrupted 512, corrupted 512], blocks of 32, the
        0.5B-class decoder's heads (12 q, 4 kv, d 128): three launches of the
        second-interval attention (attention_part_kernel then
        attention_merge_kernel each), the shapes bench.py times.

All hold a few GB on the device.  The sweep's shapes and inputs are the ones
bench.py times for its kernel roofline.
"""
from __future__ import annotations

import sys

from . import synth


def forward_gemm_shapes(cfg: synth.ModelConfig):
    """(N, K) of every GEMM launch in one decoder forward, in launch order."""
    h, f = cfg.hidden, cfg.ffn
    shapes = []
    for _ in range(cfg.n_layers):
        shapes += [(cfg.q_dim + 2 * cfg.kv_dim, h), (h, cfg.q_dim), (2 * f, h), (h, f)]
    shapes.append((cfg.vocab, h))
    return shapes


class GemmSweep:
    """Device weights, hi + lo input planes and outputs for the forward's GEMMs
    at `tokens` tokens (bf16 models), launched as the decoder launches them:
    the two-plane tcgen05 kernel, each launch with programmatic dependent
    launch so that it may start while the previous one finishes."""

    def __init__(self, cfg: synth.ModelConfig, tokens: int, device, seed: int = 0):
        import torch
        from . import gocr
        if cfg.dtype != synth.BF16:
            raise ValueError("the GEMM sweep runs the bf16 decoder's kernel")
        self.lib = gocr.load()
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.device = device
        self.tokens = tokens
        self.shapes = forward_gemm_shapes(cfg)
        self.ws = [(0.02 * torch.randn((n, k), generator=g, device=device)).to(torch.bfloat16)
                   for n, k in self.shapes]
        self.xs = {}
        for k in sorted({k for _, k in self.shapes}):
            x = torch.randn((tokens, k), generator=g, device=device)
            hi = x.to(torch.bfloat16)
            self.xs[k] = (hi, (x - hi.float()).to(torch.bfloat16))
        self.ys = [torch.empty((tokens, n), dtype=torch.float32, device=device) for n, _ in self.shapes]
        need = max(self.lib.gocr_op_linear_workspace(tokens, n, k) for n, k in self.shapes)
        self.workspace = torch.zeros(need, dtype=torch.uint8, device=device)

    def run(self):
        """Enqueue the forward's GEMM launches on the current stream."""
        import torch
        from . import gocr
        stream = torch.cuda.current_stream(self.device).cuda_stream
        for (n, k), w, y in zip(self.shapes, self.ws, self.ys):
            xh, xl = self.xs[k]
            rc = self.lib.gocr_op_linear_planes(xh.data_ptr(), xl.data_ptr(), w.data_ptr(), y.data_ptr(),
                                                self.tokens, n, k, self.workspace.data_ptr(),
                                                self.workspace.numel(), gocr.OP_OVERLAP, stream)
            if rc != gocr.GOCR_OK:
                raise gocr.GocrError(rc, gocr.last_error(None))

    def graph(self):
        """The launches captured in one CUDA graph, so that timing them
        measures the GPU and not the host's launch rate."""
        import torch
        self.run()  # tensor maps and kernel attributes are set up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        return g

    def algorithmic_bytes(self) -> float:
        """Mean bytes per launch: weights, both input planes, fp32 output."""
        T = self.tokens
        return sum(n * k * 2 + 2 * T * k * 2 + T * n * 4 for n, k in self.shapes) / len(self.shapes)


class TrainMask:
    """bf16 hi + lo planes of seeded Gaussian q [L, Hq, d], k and v [Hkv, L, d]
    and the three-stream key intervals on the device, for one attention call
    over the whole packed training sequence."""

    def __init__(self, cfg: synth.ModelConfig, device, P: int = 1024, N: int = 512, block: int = 32, seed: int = 0):
        import torch
        from . import gocr
        self.P, self.N, self.block, self.L = P, N, block, P + 3 * N
        self.cfg = cfg
        self.lim, self.lo2, self.hi2, _ = gocr.three_stream_ranges(P, N, block)
        g = torch.Generator(device="cpu").manual_seed(seed)

        def planes(shape):
            x = torch.randn(*shape, generator=g)
            hi = x.to(torch.bfloat16)
            return hi.to(device), (x - hi.float()).to(torch.bfloat16).to(device)

        self.q = planes((self.L, cfg.n_q_heads, cfg.head_dim))
        self.k = planes((cfg.n_kv_heads, self.L, cfg.head_dim))
        self.v = planes((cfg.n_kv_heads, self.L, cfg.head_dim))
        self.d_lim, self.d_lo2, self.d_hi2 = (torch.from_numpy(a).to(device) for a in (self.lim, self.lo2, self.hi2))

    def run(self):
        from . import gocr
        return gocr.op_attention(self.q, self.k, self.v, self.d_lim, gocr.DTYPE_BF16, lo2=self.d_lo2, hi2=self.d_hi2)

    def visible_pairs(self) -> int:
        """(row, key) pairs the mask lets through (both intervals)."""
        import numpy as np
        return int(np.sum(self.lim + 1) + np.sum(np.maximum(self.hi2 - self.lo2 + 1, 0)))

    def flops(self) -> float:
        """QK^T and PV multiply-adds over the visible pairs, 2 flops each."""
        return 4.0 * self.visible_pairs() * self.cfg.n_q_heads * self.cfg.head_dim


def train_mask_case():
    import torch
    tm = TrainMask(synth.BASE, torch.device("cuda:0"))
    for _ in range(3):
        tm.run()
    torch.cuda.synchronize()


def draft_case(B: int = 32):
    from . import gocr
    cfg = synth.BASE
    W = synth.make_weights(cfg)
    dec = gocr.Decoder(cfg, W, max_ctx=1024 + 2 * B + 16, max_block=B)
    del W
    dec.prefill(0, synth.make_prefix(cfg, 1024))
    _, x0 = dec.state(0)
    for _ in range(2):
        dec.debug_forward(0, gocr.FWD_DRAFT, [x0] + [0] * B)
    dec.close()


def sweep_case():
    import torch
    sw = GemmSweep(synth.BASE, 33, torch.device("cuda:0"))
    g = sw.graph()
    g.replay()
    torch.cuda.synchronize()


def batch_case():
    from . import gocr
    cfg = synth.BASE
    wl = synth.WORKLOADS["batch"]
    prefix_lens, new_lens = synth.batch_lengths(wl.n_requests)
    W = synth.make_weights(cfg)
    dec = gocr.Decoder(cfg, W, max_ctx=max(prefix_lens) + max(new_lens) + wl.block + 8, max_block=wl.block,
                       max_requests=wl.n_requests)
    del W
    for r in range(wl.n_requests):
        dec.prefill(r, synth.make_prefix(cfg, prefix_lens[r], seed=synth.REQUEST_PREFIX_SEED0 + r))
    dec.decode_batch(list(range(wl.n_requests)), gocr.MODE_SELFSPEC, wl.block, [3] * wl.n_requests)
    dec.close()


def main(argv):
    what = argv[1] if len(argv) > 1 else ""
    if what == "draft":
        draft_case(int(argv[2]) if len(argv) > 2 else 32)
    elif what == "sweep":
        sweep_case()
    elif what == "batch":
        batch_case()
    elif what == "train_mask":
        train_mask_case()
    else:
        print(__doc__)
        return 2
    print("ok")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
