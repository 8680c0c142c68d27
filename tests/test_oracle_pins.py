"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import pins
from oracle import core, dense

import numpy as np


@pytest.fixture(scope="module", autouse=True)
def _real_oracle():
    core.bind()
    yield


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(core)


def _mask_block(args):
    kv = dict(a.split("=") for a in args.split())
    return int(kv["seq_q"]), int(kv["seq_kv"]), int(kv["position_offset"])


def test_kopitiam_printed_values():
    """Every value printed in the unit tests of kopitiam-runtime src/attention.rs,
    reproduced by the dense formulation (`causal_mask`, `repeat_kv_heads`, softmax)."""
    seen = set()
    for blk in pins.golden_blocks("kopitiam_mask_and_heads.txt"):
        name = blk[0].split()[1]
        args = blk[1].partition(" ")[2]
        rows = np.array([pins._vec(r) for r in blk[2:]])
        seen.add(name)
        if name.startswith("causal_mask") or name.startswith("masked_logits"):
            m = dense.causal_mask(*_mask_block(args))[0]
            assert np.array_equal(m, rows)
            assert np.all(np.isneginf(m[rows == -np.inf]))
        elif name.startswith("masked_softmax"):
            kv = dict(a.split("=") for a in args.split())
            scores = np.array([float(x) for x in kv["scores"].split(",")])[None, None]
            probs = dense.softmax_last(scores + dense.causal_mask(1, 3, 0))[0]
            assert abs(probs[0, 0] - rows[0, 0]) < 1e-6
            assert probs[0, 1] == 0.0 and probs[0, 2] == 0.0
        elif name.startswith("repeat_kv_heads"):
            kv = dict(a.split("=") for a in args.split())
            x = np.array([float(v) for v in kv["kv"].split(",")]).reshape(
                [int(s) for s in kv["shape"].split(",")])
            out = dense.repeat_kv_heads(x, int(kv["group_size"])).reshape(-1)
            assert np.array_equal(out, rows.reshape(-1))
        else:
            raise AssertionError(name)
    assert len(seen) == 6


def test_threads_reported():
    assert core.threads() >= 1
