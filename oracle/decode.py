"""Oracle decoding loops: AR greedy (the definition) and the self-speculative round
(the algorithm, step by step).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module.

Sources (page title, section):
* GravityOCR review (euisuk-chung), §2 "Task Formulation": AR greedy decoding,
  one token per forward, top-1 (eq. 1-2).
* GravityOCR review, §3.2 "Self-Speculative Decoding", and Appendix B.2
  "Self-Speculative Decoding and KV-Cache Update" (six steps); velog review,
  "추론: 드래프트 forward 한 번 + 검증 forward 한 번" (the round and its
  acceptance rule).
* GravityOCR review, §4.1 eq. (5): tokens per forward (TPF) counts committed
  tokens over draft plus verify forwards, prefill excluded; AR has TPF 1.

Readings where the pages are silent (each listed in the design notes):
* the first output token is the argmax of the prefill's last row;
* the boundary row of the draft is causal and does not read the [M] rows;
* the [M] rows sit at consecutive positions p+1..p+B and read x0;
* the verify window has B+1 rows and yields a_1..a_{B+1};
* eos_id < 0 disables the stop token; max_new counts the prefill token and
  the last round commits only what is left;
* forced acceptance replaces d_j by the AR continuation for j <= G and makes
  d_{G+1} differ from it.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Sequence

import numpy as np

from .model import (Model, argmax_lowest, causal_mask, draft_mask, forward,
                    token_rows)


@dataclasses.dataclass
class State:
    """Per-request decode state.

    cache_k/cache_v hold the causal state of every committed token except the
    boundary token x0 (Appendix B.2, first step), so len(cache) == p and x0
    sits at position p.
    """

    cache_k: List[np.ndarray]
    cache_v: List[np.ndarray]
    x0: int
    out: List[int]

    @property
    def p(self) -> int:
        return int(self.cache_k[0].shape[0])

    def truncate(self, n: int) -> None:
        self.cache_k = [k[:n] for k in self.cache_k]
        self.cache_v = [v[:n] for v in self.cache_v]

    def append(self, new_k: Sequence[np.ndarray], new_v: Sequence[np.ndarray]) -> None:
        self.cache_k = [np.concatenate([a, b], axis=0) for a, b in zip(self.cache_k, new_k)]
        self.cache_v = [np.concatenate([a, b], axis=0) for a, b in zip(self.cache_v, new_v)]


@dataclasses.dataclass
class RoundLog:
    p: int            # cache length at round start (position of x0)
    x0: int
    a0: int
    drafts: List[int]  # d_1..d_B as verified (after any override)
    verify: List[int]  # a_1..a_{B+1}
    A: int            # accepted draft count
    committed: List[int]


def prefill(model: Model, prefix: np.ndarray) -> State:
    """Causal forward of the prefix at positions 0..P-1; the last row's argmax is out[0]."""
    P = prefix.shape[0]
    ck = [np.zeros((0, model.cfg.n_kv_heads, model.cfg.head_dim), model.dtype)
          for _ in range(model.cfg.n_layers)]
    cv = [c.copy() for c in ck]
    logits, k, v = forward(model, np.asarray(prefix, model.dtype), np.arange(P), ck, cv,
                           causal_mask(np.arange(P), P))
    t0 = int(argmax_lowest(logits[-1:])[0])
    return State(cache_k=list(k), cache_v=list(v), x0=t0, out=[t0])


def ar_forward(model: Model, st: State):
    """Forward the boundary token x0 at position p (reads keys 0..p)."""
    p = st.p
    return forward(model, token_rows(model, [st.x0]), [p], st.cache_k, st.cache_v,
                   causal_mask([p], p + 1))


def ar_step(model: Model, st: State) -> int:
    logits, k, v = ar_forward(model, st)
    st.append(k, v)
    nxt = int(argmax_lowest(logits)[0])
    st.out.append(nxt)
    st.x0 = nxt
    return nxt


def _stopped(out: Sequence[int], max_new: int, eos_id: int) -> bool:
    return len(out) >= max_new or (eos_id >= 0 and len(out) > 0 and out[-1] == eos_id)


def ar_decode(model: Model, prefix: np.ndarray, max_new: int, eos_id: int = -1) -> List[int]:
    """Greedy AR decoding, one token per forward; out counts the prefill token."""
    st = prefill(model, prefix)
    while not _stopped(st.out, max_new, eos_id):
        ar_step(model, st)
    return list(st.out)


def draft_forward(model: Model, st: State, B: int):
    """Draft forward: [x0, M x B] at positions p..p+B with the draft mask."""
    p = st.p
    rows = token_rows(model, [st.x0] + [-1] * B)
    return forward(model, rows, np.arange(p, p + B + 1), st.cache_k, st.cache_v,
                   draft_mask(p, B))


def verify_forward(model: Model, st: State, a0: int, drafts: Sequence[int]):
    """Verify forward: [a0, d1..dB] at positions p+1..p+B+1, token-causal.

    st must already hold x0's causal state at position p (the draft wrote it).
    """
    p1 = st.p
    B = len(drafts)
    rows = token_rows(model, [a0] + list(drafts))
    pos = np.arange(p1, p1 + B + 1)
    return forward(model, rows, pos, st.cache_k, st.cache_v, causal_mask(pos, p1 + B + 1))


def accept_length(drafts: Sequence[int], verify: Sequence[int]) -> int:
    """A = the largest k with d_j == a_j for every 1 <= j <= k (verify[j-1] is a_j)."""
    A = 0
    while A < len(drafts) and int(drafts[A]) == int(verify[A]):
        A += 1
    return A


Override = Callable[[int, int, List[int]], List[int]]  # (round, committed, drafts) -> drafts


def forced_override(ref: Sequence[int], schedule: Sequence[int], vocab: int) -> Override:
    """Drafts equal to the reference continuation up to G_r, then one mismatch.

    With c tokens committed at round start, d_j = ref[c + j] for 1 <= j <= G_r
    and d_{G_r + 1} = (ref[c + G_r + 1] + 1) mod V when G_r < B.  Positions past
    the end of ref keep the model's own draft.
    """
    ref = [int(t) for t in ref]

    def f(r: int, c: int, drafts: List[int]) -> List[int]:
        G = int(schedule[r]) if r < len(schedule) else 0
        B = len(drafts)
        d = list(drafts)
        for j in range(1, min(G, B) + 1):
            if c + j < len(ref):
                d[j - 1] = ref[c + j]
        if G < B and c + G + 1 < len(ref):
            d[G] = (ref[c + G + 1] + 1) % vocab
        return d

    return f


def selfspec_round(model: Model, st: State, B: int, max_new: int, eos_id: int = -1,
                   override: Optional[Override] = None, round_index: int = 0) -> RoundLog:
    """One self-speculative round (review §3.2 and Appendix B.2).

    1. Draft: x0 and B [M] rows; row 0 is causal and gives a0, rows 1..B give
       the drafts; the forward writes the causal state of x0 at position p.
    2. Verify: [a0, d1..dB] at p+1..p+B+1, causal; gives a_1..a_{B+1} and
       writes causal state over the draft's mask slots.
    3. Accept the longest prefix with d_j == a_j; commit a0, d_1..d_A,
       a_{A+1} (truncated at max_new or after the first eos).
    4. Roll back the rejected suffix: the cache keeps positions 0..p+A+1 and
       a_{A+1} becomes the next boundary.
    """
    p = st.p
    c = len(st.out)
    logits_d, kd, vd = draft_forward(model, st, B)
    am = argmax_lowest(logits_d)
    a0 = int(am[0])
    drafts = [int(t) for t in am[1:]]
    if override is not None:
        drafts = override(round_index, c, drafts)
    # Keep only x0's causal state from the draft; the [M] slots are overwritten.
    st.append([k[:1] for k in kd], [v[:1] for v in vd])
    logits_v, kv_, vv_ = verify_forward(model, st, a0, drafts)
    verify = [int(t) for t in argmax_lowest(logits_v)]
    A = accept_length(drafts, verify)
    commit = [a0] + verify[:A + 1]
    # commit a0, d_1..d_A (== a_1..a_A) and a_{A+1}, within the stop condition
    room = max_new - c
    commit = commit[:room]
    if eos_id >= 0 and eos_id in commit:
        commit = commit[: commit.index(eos_id) + 1]
    st.append(kv_, vv_)
    st.truncate(p + A + 2)
    st.out.extend(commit)
    st.x0 = verify[A]
    return RoundLog(p=p, x0=int(st.out[c - 1]), a0=a0, drafts=drafts, verify=verify, A=A,
                    committed=commit)


def selfspec_decode(model: Model, prefix: np.ndarray, B: int, max_new: int, eos_id: int = -1,
                    override: Optional[Override] = None):
    """Self-speculative decoding until max_new tokens (or eos); returns (out, round logs)."""
    st = prefill(model, prefix)
    logs = []
    r = 0
    while not _stopped(st.out, max_new, eos_id):
        logs.append(selfspec_round(model, st, B, max_new, eos_id, override, r))
        r += 1
    return list(st.out), logs


def tokens_per_forward(committed_decode: int, forwards: int) -> float:
    """Eq. (5) of the review's §4.1: committed tokens / (draft + verify forwards)."""
    return committed_decode / forwards if forwards else 0.0


def round_stats(logs: Sequence[RoundLog]) -> dict:
    """Rounds, forwards (two per round), committed tokens, accepted drafts, TPF."""
    committed = sum(len(g.committed) for g in logs)
    accepted = sum(g.A for g in logs)
    forwards = 2 * len(logs)
    return {"rounds": len(logs), "forwards": forwards, "committed": committed,
            "accepted_drafts": accepted, "tpf": tokens_per_forward(committed, forwards)}
