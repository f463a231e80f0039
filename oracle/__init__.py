"""CPU oracle for the self-speculative decode round.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this package.  The CUDA path never
calls it and shares no code with it (the seeded input generators, which hold
none of the method's arithmetic, are the only thing both sides consume).

Plain NumPy in float64 by default, with explicit dense mask matrices.
model.py: the decoder and the masks; decode.py: AR greedy and the
self-speculative round; diffusion.py: direct block-diffusion decoding and
rounds with refined drafts; sampling.py: AR sampling and the
acceptance-rejection round, with the Philox4x32-10 generator.

Parity notes: the pages print no worked numeric example (their B = 4 example
and their Figure 4 are images missing from the text), so no function here is
pinned to a printed decode trace: "parity unpinned" for a worked example.
Every function is pinned instead to closed forms, library routines, brute-force
constructions and the method's own invariants (exact AR equivalence, commit
bounds, the causal-cache invariant) in the CPU tests.
"""
from .model import (Model, argmax_lowest, attention, causal_mask, draft_mask, forward,
                    prefill_cache, rmsnorm, rope, silu, softmax_masked, three_stream_mask, token_rows,
                    top2_margin, verify_mask)
from .decode import (RoundLog, State, accept_length, ar_decode, ar_forward, ar_step,
                     draft_forward, forced_override, prefill, round_stats, selfspec_decode,
                     selfspec_round, tokens_per_forward, verify_forward)
from .diffusion import (BlockLog, RefinedRoundLog, StepLog, choose_slots, confidence,
                        diffusion_block, diffusion_decode, diffusion_stats, refined_decode,
                        refined_round, refined_stats, window_forward)
from . import sampling

__all__ = [
    "Model", "argmax_lowest", "attention", "causal_mask", "draft_mask", "forward",
    "prefill_cache", "rmsnorm", "rope", "silu", "softmax_masked", "three_stream_mask", "token_rows",
    "top2_margin",
    "verify_mask", "RoundLog", "State", "accept_length", "ar_decode", "ar_forward", "ar_step",
    "draft_forward", "forced_override", "prefill", "round_stats", "selfspec_decode",
    "selfspec_round", "tokens_per_forward", "verify_forward",
    "BlockLog", "RefinedRoundLog", "StepLog", "choose_slots", "confidence", "diffusion_block",
    "diffusion_decode", "diffusion_stats", "refined_decode", "refined_round", "refined_stats",
    "window_forward", "sampling",
]
