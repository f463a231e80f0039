"""Seeded synthetic inputs shared by the CUDA path, its tests and the oracle.

This module draws numbers and rounds them to the storage type; it holds none of
the decoding method's arithmetic.  The method is the self-speculative decode
round of a shared AR / block-diffusion decoder (GravityOCR, "Diffusion Drafts,
AR Verifies", §3.2 and Appendix B.2).  The pages ship no checkpoint and no
data, so every input here is a random stand-in with the pages' shapes:

* decoder weights N(0, 0.02) drawn in a fixed order from one seed, plus the
  single added [M] mask-token embedding row (GravityOCR review, §3.1
  "AR-to-Diffusion Conversion");
* a prefix of N(0, 1) embeddings standing in for the image + prompt prefill;
* forced-acceptance schedules: accepted-draft counts per round drawn from a
  geometric law with a stated mean (the pages' per-type acceptance, Table 4);
* ragged batched-request lengths (page-level concurrency, Appendix C).

Norm gains are ones (a gain of 0.02 would collapse the signal); the reading is
stated with the model definition in the oracle.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    """Decoder dimensions.  Every linear is stored [out, in] row-major."""

    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    dtype: str  # "f32" | "bf16"
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def weight_bytes_per_forward(self) -> int:
        """Bytes of every matrix one forward streams (norm gains excluded)."""
        es = 2 if self.dtype == BF16 else 4
        h, f = self.hidden, self.ffn
        per_layer = (self.q_dim + 2 * self.kv_dim) * h + h * self.q_dim + 2 * f * h + h * f
        return es * (self.n_layers * per_layer + self.vocab * h)

    def kv_bytes_per_token(self) -> int:
        es = 2 if self.dtype == BF16 else 4
        return es * 2 * self.n_layers * self.kv_dim


# The tiny fp32 decoder the oracle runs in full, and the 0.5B-class bf16
# decoder of the region workloads.
TINY = ModelConfig(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                   ffn=704, vocab=1024, dtype=F32)
BASE = ModelConfig(n_layers=16, hidden=1536, n_q_heads=12, n_kv_heads=4, head_dim=128,
                   ffn=4096, vocab=65536, dtype=BF16)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode workload: a model, a prefix length, a block size and a length."""

    name: str
    model: ModelConfig
    prefix_len: int
    block: int
    max_new: int
    forced_mean: Optional[float] = None  # None = natural drafts
    n_requests: int = 1


WORKLOADS: Dict[str, Workload] = {
    # tiny fp32 decoder, both modes, oracle-sized
    "tiny": Workload("tiny-fp32-prefix64-B8-new128", TINY, 64, 8, 128),
    # text-region decode: 73 output tokens is the pages' mean for text regions
    "text": Workload("text-region-bf16-0.5B-prefix1024-B32-new73", BASE, 1024, 32, 73),
    # table-region decode: 872 tokens (the pages' table mean), forced mean 9
    "table": Workload("table-region-bf16-0.5B-prefix2048-B32-new872-forced9", BASE, 2048, 32, 872,
                      forced_mean=9.0),
    # block-size sweep: B in SWEEP_BLOCKS x forced means SWEEP_MEANS, 512 tokens (headline B=32, mean 9)
    "sweep": Workload("block-sweep-bf16-0.5B-prefix2048-new512", BASE, 2048, 32, 512, forced_mean=9.0),
    # page-level batch: 16 ragged requests, B=32, per-request forced mean 9
    "batch": Workload("page-batch-bf16-0.5B-16req-ragged-B32-forced9", BASE, 0, 32, 0, forced_mean=9.0,
                      n_requests=16),
}
SWEEP_BLOCKS = (8, 16, 32, 64)
SWEEP_MEANS = (4.0, 9.0, 19.0)
BATCH_REQUESTS = 16

WEIGHT_SEED = 0
PREFIX_SEED = 1
SCHEDULE_SEED = 3
BATCH_LENGTH_SEED = 5
REQUEST_PREFIX_SEED0 = 1000


# --------------------------------------------------------------------------
# bf16 storage (round to nearest even on the host, once)
# --------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r.reshape(a.shape)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 values exactly representable in the storage dtype (fp32 array)."""
    if dtype == BF16:
        return bf16_to_f32(bf16_bits(x))
    return np.ascontiguousarray(x, dtype=np.float32)


# --------------------------------------------------------------------------
# weights, prefix, schedules
# --------------------------------------------------------------------------

LAYER_MATS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def layer_shapes(cfg: ModelConfig) -> Dict[str, tuple]:
    h, f = cfg.hidden, cfg.ffn
    return {"wq": (cfg.q_dim, h), "wk": (cfg.kv_dim, h), "wv": (cfg.kv_dim, h),
            "wo": (h, cfg.q_dim), "wg": (f, h), "wu": (f, h), "wd": (h, f)}


def make_weights(cfg: ModelConfig, seed: int = WEIGHT_SEED, std: float = 0.02) -> dict:
    """Random-init decoder, every value already representable in cfg.dtype.

    Draw order (one generator): E, m, then per layer wq wk wv wo wg wu wd, then
    the untied LM head.  Norm gains are ones.  Returns fp32 arrays.
    """
    rng = np.random.default_rng(seed)

    def draw(shape):
        a = rng.standard_normal(size=shape, dtype=np.float32)
        a *= np.float32(std)
        return round_to_storage(a, cfg.dtype)

    W = {"embed": draw((cfg.vocab, cfg.hidden)), "mask_embed": draw((cfg.hidden,))}
    shapes = layer_shapes(cfg)
    layers = []
    for _ in range(cfg.n_layers):
        lw = {name: draw(shapes[name]) for name in LAYER_MATS}
        lw["g_attn"] = np.ones(cfg.hidden, np.float32)
        lw["g_mlp"] = np.ones(cfg.hidden, np.float32)
        layers.append(lw)
    W["layers"] = layers
    W["g_final"] = np.ones(cfg.hidden, np.float32)
    W["lm_head"] = draw((cfg.vocab, cfg.hidden))
    return W


def make_prefix(cfg: ModelConfig, length: int, seed: int = PREFIX_SEED) -> np.ndarray:
    """Synthetic image+prompt prefix embeddings N(0, 1), [length, hidden]."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(size=(length, cfg.hidden), dtype=np.float32)
    return round_to_storage(a, cfg.dtype)


def accept_schedule(mean: float, n_rounds: int, seed: int = SCHEDULE_SEED) -> np.ndarray:
    """Forced accepted-draft counts G_r >= 0, geometric with E[G] = mean.

    P(G = k) = (1 - q)^k q with q = 1 / (mean + 1).  numpy's geometric counts
    trials up to the first success (support 1, 2, ...), hence the minus one.
    """
    rng = np.random.default_rng(seed)
    q = 1.0 / (mean + 1.0)
    return (rng.geometric(q, size=n_rounds) - 1).astype(np.int32)


def batch_lengths(n: int = BATCH_REQUESTS, seed: int = BATCH_LENGTH_SEED):
    """Ragged page-level requests: prefix U{512..3072}, output log-uniform 32..1024."""
    rng = np.random.default_rng(seed)
    prefix = rng.integers(512, 3073, size=n)
    new = np.rint(np.exp(rng.uniform(math.log(32), math.log(1024), size=n))).astype(np.int64)
    return [int(x) for x in prefix], [int(x) for x in new]


def random_tokens(vocab: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, vocab, size=n).astype(np.int32)


def weights_as_storage(W: dict, cfg: ModelConfig) -> dict:
    """Same tree with every array in its storage bits (uint16 for bf16, fp32 otherwise)."""
    conv = (lambda a: bf16_bits(a)) if cfg.dtype == BF16 else (lambda a: np.ascontiguousarray(a, np.float32))
    out = {k: conv(v) for k, v in W.items() if k != "layers"}
    out["layers"] = [{k: conv(v) for k, v in lw.items()} for lw in W["layers"]]
    return out


def scaled_config(cfg: ModelConfig, **kw) -> ModelConfig:
    return dataclasses.replace(cfg, **kw)

