"""Pins of the oracle's arms of the attention row: sliding window, sink logits,
logit softcap and ALiBi slopes (frink-models src/decoder/attn_block.rs,
`push_and_attend_row`: one kernel for plain, windowed, softcapped and
sink-bearing layers, plus ALiBi slopes). The pages print no formula for the
arms; the readings are stated in oracle/gqa_oracle.c. Each pin (tests/pins.py)
fixes a part of a reading by a closed form, a limit or the independent
mask-matrix form; tests/test_oracle_mutants.py checks that planted mistakes in
the arms (a window off by one, an ALiBi bias of the wrong sign, a sink left out
of the denominator, a softcap applied after the bias) each trip one."""
import numpy as np

import pins
from oracle import core


def test_arms_loops_equal_mask_matrix():
    pins.pin_arms_loops_equal_mask_matrix(core)


def test_arms_vanish_at_their_limits():
    pins.pin_arms_vanish_at_their_limits(core)


def test_arms_closed_forms():
    pins.pin_arms_closed_forms(core)


def test_softcap_bounds_the_scores():
    """With a cap c every score lies in (-c, c): a sink of logit c keeps at least
    1 / (n + 1) of the weight for n visible keys (V = 1 reads the keys' total)."""
    rng = np.random.default_rng(6)
    q = rng.standard_normal((2, 5, 4, 8)) * 50.0
    k = rng.standard_normal((2, 2, 12, 8))
    ones = np.ones((2, 2, 12, 8))
    cap, base = 0.5, [9, 12]
    mass = core.attention_arms(q, k, ones, base, 1.0, softcap=cap, sinks=[cap] * 4)
    for b in range(2):
        for i in range(5):
            n = base[b] - 5 + i + 1
            assert (mass[b, i] <= n / (n + 1) + 1e-12).all()
