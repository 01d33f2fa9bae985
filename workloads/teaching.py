"""The deterministic 27,525-token teaching input of the long-context decode page.

Source: "Why your local LLM feels dumber than it is" (Part 3.14), section
"Plugging in actual numbers".  Every token gets an already-scaled score and a
scalar value.  Both repeat with period 12; the score of a token also gets an
offset of 0.125 times (its 64-token block number mod 9).  All scores and values
are multiples of 1/8 of magnitude at most 7, so they are exact in bfloat16.

This is input data only; nothing here computes attention.
"""
from __future__ import annotations

TOKENS = 27_525
BLOCK = 64
SCORE_PATTERN = (0.5, 1.0, 0.75, -2.0, -1.25, -0.75, -0.5, -3.0, -0.25, -2.25, 0.75, 0.5)
VALUE_PATTERN = (1.875, 3.5, -0.5, 6.0, 0.0, -1.0, 5.5, -0.5, -3.5, 0.5, 4.0, -2.5)


def teaching_scores_values(tokens: int = TOKENS) -> tuple[list[float], list[float]]:
    scores, values = [], []
    period = len(SCORE_PATTERN)
    for t in range(tokens):
        block_offset = 0.125 * ((t // BLOCK) % 9)
        scores.append(SCORE_PATTERN[t % period] + block_offset)
        values.append(VALUE_PATTERN[t % period])
    return scores, values
