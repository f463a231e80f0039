"""Oracle for the block-diffusion paths of the shared decoder: direct
block-diffusion decoding, and self-speculative rounds whose draft is refined
over several denoising steps before the verify forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module.

Sources (page title, section):
* GravityOCR review (euisuk-chung), §2 "Block Diffusion": direct inference
  starts from an all-mask block, fixes chosen tokens over several steps and
  predicts the rest again; finished blocks keep their KV cache.
* GravityOCR review, Appendix B.1 "Direct Block-Diffusion Decoding": a step
  fixes every position whose confidence reaches the threshold, or the single
  most confident position when none does; a finished block needs a separate
  cache-write forward that neither checks nor replaces tokens; a finished
  block holding EOS is cut at the first EOS and decoding stops.
* Trillion Labs blog post, the confidence-threshold paragraph: confidence is
  the probability the model gives the token it predicts; only positions above
  the threshold are filled, else the one most confident position.
* GravityOCR review, Appendix D "Draft Schedule" (and the blog's "one draft is
  enough" paragraph): the draft of a self-speculative round can be refined
  over several denoising steps with a draft-side threshold before verify
  (one-shot TPF 9.00 against 6.93 with four steps).

Readings where the pages are silent (each listed in the design notes):
* the window is the self-speculative draft window: the boundary token x0 at
  position p and B slots at p+1..p+B, under the draft mask (x0 causal, the
  slots reading the cache and the whole window); a slot holds [M] until it is
  fixed, then the fixed token;
* with the shift-by-one convention (review §3.1), row r's logits predict the
  token at position p+r+1, so slot s (position p+s) takes row s-1's argmax,
  and row B's prediction lies past the block;
* confidence = the largest softmax probability of the row;
* ties in "most confident" go to the lowest slot index; a confidence equal to
  the threshold passes it;
* the cache-write forward is token-causal over [x0, y_1..y_B] at p..p+B (the
  verify window's shape); the cache then keeps positions 0..p+B-1 and y_B is
  the next boundary; it is skipped when decoding stops with the block;
* a block is finished before max_new or EOS truncation, like the EOS cut;
* TPF counts every forward: denoising steps and cache writes;
* refined drafts: a round runs at most n_steps draft forwards; slots fixed in
  a step keep their token; after the last step the verify window is
  [a0 = slot 1, slots 2..B, row B's prediction], unfixed slots taking the last
  step's predictions; verify, accept and rollback are the one-shot round's.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np

from .decode import State, _stopped, accept_length, prefill, verify_forward
from .model import Model, argmax_lowest, causal_mask, draft_mask, forward, token_rows, top2_margin


def confidence(logits: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per row: (argmax token, largest softmax probability).

    The largest probability is exp(l_max) / sum_v exp(l_v) = 1 / sum_v exp(l_v - l_max).
    """
    tok = argmax_lowest(logits)
    lg = np.asarray(logits, dtype=np.float64)
    m = lg.max(axis=-1, keepdims=True)
    conf = 1.0 / np.sum(np.exp(lg - m), axis=-1)
    return tok, conf


def choose_slots(conf: Sequence[float], masked: Sequence[int], tau: float) -> List[int]:
    """The slots one denoising step fixes (review Appendix B.1; blog, threshold).

    Every still-masked slot whose confidence is at least tau; if there is none,
    the most confident masked slot alone (the lowest index among equals).
    """
    passed = [s for s in masked if conf[s] >= tau]
    if passed:
        return passed
    best = None
    for s in masked:
        if best is None or conf[s] > conf[best]:
            best = s
    return [] if best is None else [best]


def window_forward(model: Model, st: State, slots: Sequence[int]):
    """Draft-window forward: x0 at p, slot s (token or -1 = [M]) at p+s, draft mask."""
    p = st.p
    B = len(slots)
    rows = token_rows(model, [st.x0] + list(slots))
    return forward(model, rows, np.arange(p, p + B + 1), st.cache_k, st.cache_v, draft_mask(p, B))


@dataclasses.dataclass
class StepLog:
    fixed: List[int]          # slot indices (0-based: slot s+1) fixed by this step
    tokens: List[int]         # the B slot predictions of the step (rows 0..B-1)
    conf: List[float]         # their confidences
    margin: List[float]       # top-two logit margin of every row of the window (diagnostic)


@dataclasses.dataclass
class BlockLog:
    p: int                    # cache length at block start (position of x0)
    x0: int
    steps: List[StepLog]
    block: List[int]          # y_1..y_B
    committed: List[int]
    cache_write: bool         # whether the cache-write forward ran


def diffusion_block(model: Model, st: State, B: int, tau: float, max_new: int,
                    eos_id: int = -1) -> BlockLog:
    """One block of direct block-diffusion decoding (review §2 and Appendix B.1).

    1. Start from B masked slots after the boundary token.
    2. Repeat: forward the window; every masked slot gets its row's argmax and
       confidence; fix the slots that reach tau, else the most confident one.
    3. When no slot is masked, commit y_1..y_B (cut at max_new and after the
       first EOS); unless decoding stops, run the causal cache-write forward
       and make y_B the next boundary.
    """
    p, x0 = st.p, st.x0
    c = len(st.out)
    slots = [-1] * B
    steps: List[StepLog] = []
    while any(s < 0 for s in slots):
        logits, _, _ = window_forward(model, st, slots)
        tok, conf = confidence(logits[:B])
        masked = [s for s in range(B) if slots[s] < 0]
        fixed = choose_slots(conf, masked, tau)
        for s in fixed:
            slots[s] = int(tok[s])
        steps.append(StepLog(fixed=fixed, tokens=[int(t) for t in tok], conf=[float(x) for x in conf],
                             margin=[top2_margin(r) for r in logits]))
    commit = list(slots)[: max_new - c]
    if eos_id >= 0 and eos_id in commit:
        commit = commit[: commit.index(eos_id) + 1]
    st.out.extend(commit)
    stop = _stopped(st.out, max_new, eos_id)
    if not stop:
        rows = token_rows(model, [x0] + slots)
        pos = np.arange(p, p + B + 1)
        _, k, v = forward(model, rows, pos, st.cache_k, st.cache_v, causal_mask(pos, p + B + 1))
        st.append(k, v)
        st.truncate(p + B)
        st.x0 = slots[B - 1]
    return BlockLog(p=p, x0=x0, steps=steps, block=list(slots), committed=commit, cache_write=not stop)


def diffusion_decode(model: Model, prefix: np.ndarray, B: int, tau: float, max_new: int,
                     eos_id: int = -1):
    """Direct block-diffusion decoding until max_new tokens or EOS; returns (out, block logs).

    out counts the prefill token, as in the AR and self-speculative loops.
    """
    st = prefill(model, prefix)
    logs = []
    while not _stopped(st.out, max_new, eos_id):
        logs.append(diffusion_block(model, st, B, tau, max_new, eos_id))
    return list(st.out), logs


def diffusion_stats(logs: Sequence[BlockLog]) -> dict:
    """Blocks, forwards (denoising steps plus cache writes), committed tokens, TPF."""
    fwd = sum(len(g.steps) + (1 if g.cache_write else 0) for g in logs)
    committed = sum(len(g.committed) for g in logs)
    return {"blocks": len(logs), "forwards": fwd, "committed": committed,
            "tpf": committed / fwd if fwd else 0.0}


# --------------------------------------------------------------------------
# self-speculative rounds with a refined draft (review Appendix D)
# --------------------------------------------------------------------------

@dataclasses.dataclass
class RefinedRoundLog:
    p: int
    x0: int
    steps: List[StepLog]
    a0: int
    drafts: List[int]         # d_1..d_B as verified
    verify: List[int]         # a_1..a_{B+1}
    A: int
    committed: List[int]


def refined_round(model: Model, st: State, B: int, tau_d: float, n_steps: int, max_new: int,
                  eos_id: int = -1) -> RefinedRoundLog:
    """One self-speculative round whose draft runs up to n_steps denoising steps.

    Each step forwards the window and fixes slots by the threshold rule with the
    draft-side threshold tau_d.  After the last step (or when no slot is left
    masked) the verify window is [slot 1 .. slot B, row B's prediction], where
    slot 1 is a0 (row 0 is causal, so its prediction never depends on the
    slots) and every unfixed slot takes the last step's prediction.  Verify,
    accept, commit and rollback are those of the one-shot round.
    """
    p, x0 = st.p, st.x0
    c = len(st.out)
    slots = [-1] * B
    steps: List[StepLog] = []
    last = None
    kd = vd = None
    for _ in range(max(1, n_steps)):
        logits, kd, vd = window_forward(model, st, slots)
        tok, conf = confidence(logits)
        last = [int(t) for t in tok]
        masked = [s for s in range(B) if slots[s] < 0]
        fixed = choose_slots(conf[:B], masked, tau_d)
        for s in fixed:
            slots[s] = last[s]
        steps.append(StepLog(fixed=fixed, tokens=last[:B], conf=[float(x) for x in conf[:B]],
                             margin=[top2_margin(r) for r in logits]))
        if all(s >= 0 for s in slots):
            break
    window = [slots[s] if slots[s] >= 0 else last[s] for s in range(B)] + [last[B]]
    a0, drafts = window[0], window[1:]
    # x0's causal state (row 0 of any step; the draft mask keeps it causal)
    st.append([k[:1] for k in kd], [v[:1] for v in vd])
    logits_v, kv_, vv_ = verify_forward(model, st, a0, drafts)
    verify = [int(t) for t in argmax_lowest(logits_v)]
    A = accept_length(drafts, verify)
    commit = ([a0] + verify[:A + 1])[: max_new - c]
    if eos_id >= 0 and eos_id in commit:
        commit = commit[: commit.index(eos_id) + 1]
    st.append(kv_, vv_)
    st.truncate(p + A + 2)
    st.out.extend(commit)
    st.x0 = verify[A]
    return RefinedRoundLog(p=p, x0=x0, steps=steps, a0=a0, drafts=drafts, verify=verify, A=A,
                           committed=commit)


def refined_decode(model: Model, prefix: np.ndarray, B: int, tau_d: float, n_steps: int,
                   max_new: int, eos_id: int = -1):
    """Self-speculative decoding with refined drafts; returns (out, round logs)."""
    st = prefill(model, prefix)
    logs = []
    while not _stopped(st.out, max_new, eos_id):
        logs.append(refined_round(model, st, B, tau_d, n_steps, max_new, eos_id))
    return list(st.out), logs


def refined_stats(logs: Sequence[RefinedRoundLog]) -> dict:
    """Rounds, forwards (draft steps plus one verify per round), committed tokens, TPF."""
    fwd = sum(len(g.steps) + 1 for g in logs)
    committed = sum(len(g.committed) for g in logs)
    return {"rounds": len(logs), "forwards": fwd, "committed": committed,
            "accepted_drafts": sum(g.A for g in logs), "tpf": committed / fwd if fwd else 0.0}
