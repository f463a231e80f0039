"""Oracle for the sampling variant: AR sampling (the definition) and the
self-speculative round with the standard speculative acceptance-rejection
rule (the algorithm).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module.

Sources (page title, section):
* GravityOCR review (euisuk-chung), §2 "Speculative Decoding": describes,
  besides the greedy top-1 verification GravityOCR uses, the standard
  stochastic acceptance-rejection rule; GravityOCR's equality claims are for
  top-1.
* Trillion Labs blog post, the paragraph on AR equivalence: with sampling the
  speculative rejection rule preserves the AR distribution.

The rule (as speculative sampling states it): a drafted token d with draft
probability q(d) and target probability p(d) is accepted with probability
min(1, p(d) / q(d)); at the first rejection a replacement is drawn from
max(0, p - q) renormalised, and the round stops; if every draft is accepted a
bonus token is drawn from the next target distribution.

Readings where the pages are silent (each listed in the design notes):
* p and q are softmax(logits / T) of the verify and draft rows, one
  temperature T > 0 for both;
* the prefill token stays the greedy argmax (the prefill call takes no
  sampling options); decode tokens are sampled;
* the boundary row's distribution is the AR target, so a0 is drawn from it
  and committed as in the greedy round;
* random numbers come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
  "Parallel random numbers: as easy as 1, 2, 3", SC 2011), which both sides
  implement from that definition: key (seed low, seed high word) and counter
  (v / 4, position, purpose, request), lane v % 4; a draw from a
  distribution is a Gumbel-max over the vocabulary with uniforms
  u = ((x >> 9) + 0.5) / 2^23 (exact in fp32, so both sides take the same
  value: a 25-bit uniform rounds near 1, where -log(-log u) is steep); purposes: 0 target token at its position
  (AR steps, a0, the bonus), 1 draft token, 2 the acceptance uniform (v = 0),
  3 the replacement after a rejection.  The token at absolute position t uses
  position t.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

from .decode import State, _stopped, draft_forward, prefill
from .model import Model, causal_mask, forward, token_rows

M32 = 0xFFFFFFFF
PHILOX_M = (0xD2511F53, 0xCD9E8D57)
PHILOX_W = (0x9E3779B9, 0xBB67AE85)
PURPOSE_TARGET, PURPOSE_DRAFT, PURPOSE_ACCEPT, PURPOSE_RESIDUAL = 0, 1, 2, 3


def philox4x32_10(ctr: np.ndarray, key: Sequence[int]) -> np.ndarray:
    """Philox4x32 with 10 rounds on counters ctr [n, 4] (uint32) and one key.

    A round multiplies word 0 and word 2 by the two multipliers, keeps the
    128-bit products' halves, and mixes them with words 1 and 3 and the key:
    (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the
    key is bumped by the two Weyl constants between rounds.
    """
    c = np.asarray(ctr, dtype=np.uint64).reshape(-1, 4) & M32
    c0, c1, c2, c3 = c[:, 0].copy(), c[:, 1].copy(), c[:, 2].copy(), c[:, 3].copy()
    k0, k1 = int(key[0]) & M32, int(key[1]) & M32
    for r in range(10):
        p0 = c0 * np.uint64(PHILOX_M[0])
        p1 = c2 * np.uint64(PHILOX_M[1])
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(M32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(M32)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0)), lo1, (hi0 ^ c3 ^ np.uint64(k1)), lo0
        if r < 9:
            k0 = (k0 + PHILOX_W[0]) & M32
            k1 = (k1 + PHILOX_W[1]) & M32
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


def uniforms(seed: int, req: int, pos: int, purpose: int, n: int) -> np.ndarray:
    """n uniforms in (0, 1) for vocabulary entries 0..n-1 of one draw."""
    blocks = (n + 3) // 4
    ctr = np.zeros((blocks, 4), np.uint64)
    ctr[:, 0] = np.arange(blocks, dtype=np.uint64)
    ctr[:, 1] = pos & M32
    ctr[:, 2] = purpose & M32
    ctr[:, 3] = req & M32
    x = philox4x32_10(ctr, (seed & M32, (seed >> 32) & M32)).reshape(-1)[:n].astype(np.float64)
    return (np.floor(x / 512.0) + 0.5) / float(1 << 23)


def gumbel_argmax(scores: np.ndarray, u: np.ndarray, diag: Optional[list] = None) -> int:
    """argmax over v of scores[v] - log(-log u[v]) (lowest index among equals);
    entries at -inf are never chosen.  With scores = log-probabilities (up to a
    constant) this is a draw from that distribution.  diag (optional) receives
    the gap between the two largest perturbed scores (a diagnostic)."""
    g = np.asarray(scores, np.float64) - np.log(-np.log(u))
    if diag is not None:
        top = np.sort(g[np.isfinite(g)])
        diag.append(float(top[-1] - top[-2]) if top.size > 1 else np.inf)
    return int(np.argmax(g))


def probs(logits_row: np.ndarray, T: float) -> np.ndarray:
    z = np.asarray(logits_row, np.float64) / T
    z = np.exp(z - z.max())
    return z / z.sum()


def sample_target(logits_row, T, seed, req, pos, diag: Optional[list] = None) -> int:
    u = uniforms(seed, req, pos, PURPOSE_TARGET, len(logits_row))
    return gumbel_argmax(np.asarray(logits_row, np.float64) / T, u, diag)


def ar_sample_decode(model: Model, prefix: np.ndarray, max_new: int, T: float, seed: int, req: int = 0,
                     eos_id: int = -1, diag: Optional[list] = None) -> List[int]:
    """AR sampling: the token at position t drawn from softmax(logits / T) of
    the row at t - 1 (the prefill token is the greedy argmax).  diag
    (optional) receives each draw's top-two perturbed-score gap."""
    st = prefill(model, prefix)
    while not _stopped(st.out, max_new, eos_id):
        p = st.p
        logits, k, v = forward(model, token_rows(model, [st.x0]), [p], st.cache_k, st.cache_v,
                               causal_mask([p], p + 1))
        st.append(k, v)
        t = sample_target(logits[0], T, seed, req, p + 1, diag)
        st.out.append(t)
        st.x0 = t
    return list(st.out)


@dataclasses.dataclass
class SampleRoundLog:
    p: int
    a0: int
    drafts: List[int]
    accept_u: List[float]     # acceptance uniform of each draft position
    ratio: List[float]        # p(d_j) / q(d_j) for the drafts examined
    A: int                    # accepted drafts
    last: int                 # the replacement (A < B) or the bonus (A = B)
    committed: List[int]
    margin: float = np.inf    # smallest top-two perturbed-score gap of the round's draws (diagnostic)
    accept_gap: float = np.inf  # smallest |u_j - min(1, ratio_j)| of the examined drafts (diagnostic)


def accept_reject(drafts: Sequence[int], q_rows: np.ndarray, p_rows: np.ndarray, u_acc: Sequence[float]):
    """The acceptance-rejection walk over one round's drafts.

    d_j (j = 1..B) is accepted when u_j < p_j(d_j) / q_j(d_j) (always when the
    ratio is at least 1); q_rows[j-1] and p_rows[j-1] are its draft and target
    distributions.  Returns (A, ratios of the examined drafts)."""
    A = 0
    ratios = []
    for j, d in enumerate(drafts):
        r = float(p_rows[j][d] / q_rows[j][d])
        ratios.append(r)
        if u_acc[j] < min(1.0, r):
            A += 1
        else:
            break
    return A, ratios


def residual_sample(p_row: np.ndarray, q_row: np.ndarray, u: np.ndarray, diag: Optional[list] = None) -> int:
    """A draw from max(0, p - q) renormalised (Gumbel-max over its log); from
    p itself when rounding leaves max(0, p - q) without mass."""
    w = np.maximum(0.0, np.asarray(p_row, np.float64) - np.asarray(q_row, np.float64))
    if not (w > 0).any():
        w = np.asarray(p_row, np.float64)
    with np.errstate(divide="ignore"):
        return gumbel_argmax(np.log(w), u, diag)


def selfspec_sample_round(model: Model, st: State, B: int, max_new: int, T: float, seed: int, req: int = 0,
                          eos_id: int = -1) -> SampleRoundLog:
    """One self-speculative round with sampling.

    Draft: a0 from the boundary row (the AR target for position p+1), d_j from
    [M] row j (draft distribution q_j for position p+1+j).  Verify [a0, d_1..d_B]:
    row j-1 gives the target p_j for position p+1+j, row B the target for
    p+B+2.  Accept-reject the drafts in order; commit a0, the accepted drafts
    and the replacement (or the bonus).  Rollback as in the greedy round.
    """
    p = st.p
    c = len(st.out)
    V = model.cfg.vocab
    lg_d, kd, vd = draft_forward(model, st, B)
    gaps: list = []
    a0 = sample_target(lg_d[0], T, seed, req, p + 1, gaps)
    drafts = [gumbel_argmax(lg_d[j] / T, uniforms(seed, req, p + 1 + j, PURPOSE_DRAFT, V), gaps)
              for j in range(1, B + 1)]
    st.append([k[:1] for k in kd], [v[:1] for v in vd])
    rows = token_rows(model, [a0] + drafts)
    pos = np.arange(p + 1, p + B + 2)
    lg_v, kv_, vv_ = forward(model, rows, pos, st.cache_k, st.cache_v, causal_mask(pos, p + B + 2))
    q_rows = np.stack([probs(lg_d[j], T) for j in range(1, B + 1)])
    p_rows = np.stack([probs(lg_v[j], T) for j in range(0, B)])
    u_acc = [float(uniforms(seed, req, p + 1 + j, PURPOSE_ACCEPT, 1)[0]) for j in range(1, B + 1)]
    A, ratios = accept_reject(drafts, q_rows, p_rows, u_acc)
    if A < B:
        last = residual_sample(p_rows[A], q_rows[A], uniforms(seed, req, p + 2 + A, PURPOSE_RESIDUAL, V), gaps)
    else:
        last = sample_target(lg_v[B], T, seed, req, p + B + 2, gaps)
    acc_gap = min((abs(u_acc[j] - min(1.0, ratios[j])) for j in range(len(ratios))), default=np.inf)
    commit = ([a0] + drafts[:A] + [last])[: max_new - c]
    if eos_id >= 0 and eos_id in commit:
        commit = commit[: commit.index(eos_id) + 1]
    st.append(kv_, vv_)
    st.truncate(p + A + 2)
    st.out.extend(commit)
    st.x0 = last
    return SampleRoundLog(p=p, a0=a0, drafts=drafts, accept_u=u_acc, ratio=ratios, A=A, last=last,
                          committed=commit, margin=min(gaps), accept_gap=acc_gap)


def selfspec_sample_decode(model: Model, prefix: np.ndarray, B: int, max_new: int, T: float, seed: int,
                           req: int = 0, eos_id: int = -1):
    """Self-speculative decoding with sampling; returns (out, round logs)."""
    st = prefill(model, prefix)
    logs = []
    while not _stopped(st.out, max_new, eos_id):
        logs.append(selfspec_sample_round(model, st, B, max_new, T, seed, req, eos_id))
    return list(st.out), logs
