"""Oracle decoder forward: plain NumPy, float64 by default, explicit mask matrices.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module; it
is the slow, obviously-correct CPU statement of what the CUDA path computes and
it shares no code with it.

The pages (GravityOCR: "Diffusion Drafts, AR Verifies"; the euisuk-chung
review, the velog review and the Trillion Labs blog post) describe the decoder
only as a pretrained AR OCR decoder plus one [M] embedding row shared by both
paths (review §3.1 "AR-to-Diffusion Conversion").  They print no architecture.
The plainest decoder consistent with the stated dimensions is used, and each
choice is a reading:

* pre-norm blocks: x += Attn(RMSNorm(x)); x += MLP(RMSNorm(x));
* RMSNorm y = x / sqrt(mean(x^2) + eps) * g, eps = 1e-6;
* every linear y = x W^T with W stored [out, in], no biases;
* rotate-half RoPE on all head dims, theta = 1e4, at absolute positions; the
  cache stores rotated keys;
* grouped-query attention: q head h reads kv head floor(h * Hkv / Hq),
  softmax(q k^T / sqrt(d)) with masked entries at -inf;
* SwiGLU MLP: (silu(x Wg^T) * (x Wu^T)) Wd^T with silu(z) = z * sigmoid(z);
* logits = RMSNorm(x; g_final) Wlm^T with an untied LM head;
* the logit at position i predicts the token at i + 1 (review §3.1, the
  shift-by-one convention shared by both paths).
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np


# --------------------------------------------------------------------------
# components
# --------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2, last axis) + eps) * g."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of x[n, H, d] at integer positions pos[n].

    Dimension i < d/2 is paired with i + d/2 and the pair is turned by the
    angle pos * theta^(-2i/d).
    """
    n, H, d = x.shape
    half = d // 2
    inv_freq = theta ** (-(np.arange(half, dtype=np.float64) * 2.0) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos = np.cos(ang)[:, None, :].astype(x.dtype)
    sin = np.sin(ang)[:, None, :].astype(x.dtype)
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def softmax_masked(s: np.ndarray, allowed: np.ndarray) -> np.ndarray:
    """Row softmax of s with disallowed entries at -inf (each row keeps >= 1 entry)."""
    s = np.where(allowed, s, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, allowed: np.ndarray) -> np.ndarray:
    """Grouped-query attention with an explicit boolean mask.

    q [n, Hq, d]; k, v [nk, Hkv, d]; allowed [n, nk] (True = query may read key).
    Returns o [n, Hq, d].
    """
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    o = np.empty_like(q)
    scale = 1.0 / math.sqrt(d)
    for h in range(Hq):
        kvh = (h * Hkv) // Hq
        s = (q[:, h, :] @ k[:, kvh, :].T) * scale
        p = softmax_masked(s, allowed)
        o[:, h, :] = p @ v[:, kvh, :]
    return o


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Per-row argmax taking the lowest index among equal maxima.  NaN is an error."""
    if np.isnan(logits).any():
        raise FloatingPointError("NaN in logits")
    return np.argmax(logits, axis=-1).astype(np.int64)


# --------------------------------------------------------------------------
# masks (rows = the window's queries, columns = absolute key positions)
# --------------------------------------------------------------------------

def causal_mask(row_pos: Sequence[int], n_keys: int) -> np.ndarray:
    """Row at absolute position t may read keys 0..t."""
    rp = np.asarray(row_pos, dtype=np.int64)[:, None]
    return np.arange(n_keys, dtype=np.int64)[None, :] <= rp


def draft_mask(p: int, B: int) -> np.ndarray:
    """Draft window [x0, M x B] at positions p..p+B over keys 0..p+B.

    The boundary row (x0 at p) is causal: keys 0..p.  Each [M] row reads the
    whole cache and the whole window, bidirectionally: keys 0..p+B (review §3.2;
    velog review, "draft forward": mask positions attend causally to the cache
    and bidirectionally inside the window).
    """
    n_keys = p + B + 1
    m = np.zeros((B + 1, n_keys), dtype=bool)
    m[0, : p + 1] = True
    m[1:, :] = True
    return m


def verify_mask(p: int, B: int) -> np.ndarray:
    """Verify window [a0, d1..dB] at positions p+1..p+B+1, token-causal."""
    return causal_mask(np.arange(p + 1, p + B + 2), p + B + 2)


def three_stream_mask(P: int, N: int, B: int) -> np.ndarray:
    """Attention mask of the joint AR / block-diffusion training forward over
    the packed sequence [prefix (P), clean response (N), corrupted stream 1
    (N), corrupted stream 2 (N)] (review §3.1 "Joint AR-Diffusion Training";
    the blog's three-stream figure).

    Rows and columns index the packed sequence.  Written from the rule text,
    entry by entry:
    * the prefix (image and prompt, never corrupted) is causal;
    * the clean stream sees the prefix and its own earlier tokens (causal);
    * a token of block b of a corrupted stream sees the prefix, the clean
      blocks before b, and every token of its own block b of its own stream
      (bidirectional inside the block); not clean block b or later, not its
      stream's other blocks, not the other corrupted stream.
    """
    L = P + 3 * N
    m = np.zeros((L, L), dtype=bool)

    def where(r):
        if r < P:
            return "prefix", r, -1
        s, i = divmod(r - P, N)
        return ("clean" if s == 0 else f"corrupt{s}"), i, i // B

    for q in range(L):
        qs, qi, qb = where(q)
        for k in range(L):
            ks, ki, kb = where(k)
            if qs == "prefix":
                ok = ks == "prefix" and k <= q
            elif qs == "clean":
                ok = ks == "prefix" or (ks == "clean" and ki <= qi)
            else:
                ok = ks == "prefix" or (ks == "clean" and kb < qb) or (ks == qs and kb == qb)
            m[q, k] = ok
    return m


# --------------------------------------------------------------------------
# forward over a window of rows, given the cache for keys before the window
# --------------------------------------------------------------------------

class Model:
    """Decoder weights in the oracle's working precision."""

    def __init__(self, W: dict, cfg, dtype=np.float64):
        self.cfg = cfg
        self.dtype = dtype
        cv = lambda a: np.asarray(a, dtype=dtype)
        self.embed = cv(W["embed"])
        self.mask_embed = cv(W["mask_embed"])
        self.g_final = cv(W["g_final"])
        self.lm_head = cv(W["lm_head"])
        self.layers = [{k: cv(v) for k, v in lw.items()} for lw in W["layers"]]


def forward(model: Model, x: np.ndarray, pos: Sequence[int],
            cache_k: List[np.ndarray], cache_v: List[np.ndarray],
            allowed: np.ndarray) -> Tuple[np.ndarray, List[np.ndarray], List[np.ndarray]]:
    """One decoder forward over the rows x[n, hidden] at absolute positions pos.

    cache_k[l], cache_v[l]: [p0, Hkv, d] keys/values of absolute positions
    0..p0-1 (rotated keys).  The window's own keys are appended after them, so
    allowed has shape [n, p0 + n] over absolute key positions 0..p0+n-1 and the
    window must sit at positions p0..p0+n-1.
    Returns (logits [n, vocab], new_k per layer [n, Hkv, d], new_v per layer).
    """
    cfg = model.cfg
    dt = model.dtype
    n = x.shape[0]
    pos = np.asarray(pos, dtype=np.int64)
    Hq, Hkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    x = np.asarray(x, dtype=dt).copy()
    new_k, new_v = [], []
    for l, lw in enumerate(model.layers):
        xn = rmsnorm(x, lw["g_attn"], cfg.rms_eps)
        q = (xn @ lw["wq"].T).reshape(n, Hq, d)
        k = (xn @ lw["wk"].T).reshape(n, Hkv, d)
        v = (xn @ lw["wv"].T).reshape(n, Hkv, d)
        q = rope(q, pos, cfg.rope_theta)
        k = rope(k, pos, cfg.rope_theta)
        new_k.append(k)
        new_v.append(v)
        K = np.concatenate([np.asarray(cache_k[l], dtype=dt), k], axis=0)
        V = np.concatenate([np.asarray(cache_v[l], dtype=dt), v], axis=0)
        o = attention(q, K, V, allowed).reshape(n, Hq * d)
        x = x + o @ lw["wo"].T
        xn = rmsnorm(x, lw["g_mlp"], cfg.rms_eps)
        hdn = silu(xn @ lw["wg"].T) * (xn @ lw["wu"].T)
        x = x + hdn @ lw["wd"].T
    logits = rmsnorm(x, model.g_final, cfg.rms_eps) @ model.lm_head.T
    return logits, new_k, new_v


def token_rows(model: Model, tokens: Sequence[int]) -> np.ndarray:
    """Embedding rows; token -1 stands for the [M] mask token."""
    rows = []
    for t in tokens:
        rows.append(model.mask_embed if int(t) < 0 else model.embed[int(t)])
    return np.stack(rows, axis=0)


def empty_cache(model: Model) -> Tuple[List[np.ndarray], List[np.ndarray]]:
    cfg = model.cfg
    z = lambda: np.zeros((0, cfg.n_kv_heads, cfg.head_dim), dtype=model.dtype)
    return [z() for _ in range(cfg.n_layers)], [z() for _ in range(cfg.n_layers)]


def prefill_cache(model: Model, prefix: np.ndarray, tokens: Sequence[int] = ()
                  ) -> Tuple[np.ndarray, List[np.ndarray], List[np.ndarray]]:
    """Causal forward of [prefix embeddings, embeddings of tokens] from position 0.

    Returns (logits, K per layer, V per layer) for all rows.
    """
    rows = np.asarray(prefix, dtype=model.dtype)
    if len(tokens):
        rows = np.concatenate([rows, token_rows(model, tokens)], axis=0)
    n = rows.shape[0]
    ck, cv = empty_cache(model)
    logits, k, v = forward(model, rows, np.arange(n), ck, cv, causal_mask(np.arange(n), n))
    return logits, k, v


def top2_margin(logits_row: np.ndarray) -> float:
    """Gap between the largest and second-largest logit (the pages' tie diagnostic)."""
    s = np.sort(np.asarray(logits_row, dtype=np.float64))
    return float(s[-1] - s[-2])


def as_model(W: dict, cfg, dtype=np.float64) -> Model:
    return W if isinstance(W, Model) else Model(W, cfg, dtype)

