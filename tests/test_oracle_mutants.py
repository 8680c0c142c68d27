"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
each one trips at least one pin. A pin set that a mistake slips through is not
pinning that part of the oracle."""
import os
import subprocess
import tempfile
import types

import numpy as np

import pytest

import pins
from oracle import core

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "gqa_oracle.c")

# (name, text in gqa_oracle.c, replacement). Each replacement keeps every memory
# access inside its buffer, so a mutant can only give wrong numbers.
MUTANTS = [
    ("head mapping h % Hkv", "int kvh = h / G;", "int kvh = h % s->Hkv;"),
    ("causal: own position excluded", "int n = base_len[b] - seq_q + i + 1;",
     "int n = base_len[b] - seq_q + i + (i > 0 ? 0 : 1);"),
    ("causal: row index ignored", "int n = base_len[b] - seq_q + i + 1;",
     "int n = base_len[b] - seq_q + 1;"),
    ("scale divides", "w[j] = scale * dot;", "w[j] = (scale != 0.0 ? dot / scale : dot);"),
    ("scale dropped", "w[j] = scale * dot;", "w[j] = dot;"),
    ("no normalisation", "out[c] = num / den;", "out[c] = num;"),
    ("value rows reversed", "num += w[j] * ld(s->v, row_index(s, b, kvh, j, s->dv, c), s->et);",
     "num += w[j] * ld(s->v, row_index(s, b, kvh, n - 1 - j, s->dv, c), s->et);"),
    ("value columns reversed", "num += w[j] * ld(s->v, row_index(s, b, kvh, j, s->dv, c), s->et);",
     "num += w[j] * ld(s->v, row_index(s, b, kvh, j, s->dv, s->dv - 1 - c), s->et);"),
    ("paged: rows reversed in block", "+ (j % s->bs)) * (size_t)d + c;",
     "+ (s->bs - 1 - j % s->bs)) * (size_t)d + c;"),
    ("rope: sign flipped", "x0 * cos(a) - x1 * sin(a)", "x0 * cos(a) + x1 * sin(a)"),
    ("rope: exponent over pairs", "pow(theta, -2.0 * pr / rot_dim)", "pow(theta, -1.0 * pr / rot_dim)"),
    ("rope: half-split pairs", "double x0 = ld(x, row + 2 * pr, et), x1 = ld(x, row + 2 * pr + 1, et);\n"
     "          st(x, row + 2 * pr, et, x0 * cos(a) - x1 * sin(a));\n"
     "          st(x, row + 2 * pr + 1, et, x0 * sin(a) + x1 * cos(a));",
     "double x0 = ld(x, row + pr, et), x1 = ld(x, row + pr + rot_dim / 2, et);\n"
     "          st(x, row + pr, et, x0 * cos(a) - x1 * sin(a));\n"
     "          st(x, row + pr + rot_dim / 2, et, x0 * sin(a) + x1 * cos(a));"),
    ("append: rotated at p+1", "int32_t pos = p;", "int32_t pos = p + 1;"),
    ("append: next slot", "size_t dst_k = (((size_t)blk * Hkv + kvh) * bs + p % bs) * (size_t)dk;",
     "size_t dst_k = (((size_t)blk * Hkv + kvh) * bs + (p + 1) % bs) * (size_t)dk;"),
    ("append: length not advanced", "seq_lens_out[b] = p + 1;", "seq_lens_out[b] = p;"),
    ("bf16: truncating round", "double r = nearbyint(ldexp(ax, -shift));",
     "double r = floor(ldexp(ax, -shift));"),
    ("bf16: ties away from zero", "double r = nearbyint(ldexp(ax, -shift));",
     "double r = round(ldexp(ax, -shift));"),
    ("bf16: widened with a shift of 15", "uint32_t u = (uint32_t)h << 16;",
     "uint32_t u = (uint32_t)h << 15;"),
    ("arms: ALiBi sign flipped", "sj += slope * (double)(j - p);", "sj += slope * (double)(p - j);"),
    ("arms: sink left out of the denominator", "double total = sink ? exp(*sink - m) : 0.0;", "double total = 0.0;"),
    ("arms: window one key wider", "int lo = (window > 0 && pos - window + 1 > 0) ? pos - window + 1 : 0;",
     "int lo = (window > 0 && pos - window > 0) ? pos - window : 0;"),
    ("arms: softcap after the bias", "if (softcap > 0.0) sj = softcap * tanh(sj / softcap);\n    sj += slope * (double)(j - p);",
     "sj += slope * (double)(j - p);\n    if (softcap > 0.0) sj = softcap * tanh(sj / softcap);"),
]


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d
    core.bind()  # back to the real oracle


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant_dir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
    path = os.path.join(mutant_dir, f"m{MUTANTS.index((name, old, new))}")
    open(path + ".c", "w").write(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", path + ".so",
                    path + ".c", "-lm"], check=True)
    core.bind(path + ".so")
    try:
        failed = []
        for pin in pins.ALL_PINS:
            try:
                pin(core)
            except (AssertionError, ValueError, FloatingPointError):
                failed.append(pin.__name__)
        assert failed, f"planted mistake '{name}' passed every pin"
    finally:
        core.bind()


# Planted mistakes in the absorbed-MLA functions of oracle/core.py (numpy, so
# each is a replacement function, handed to the pins through a stand-in module).
def _absorb_rope_dropped(q, k_b, d_nope):
    out = core.mla_absorb_q(q, k_b, d_nope)
    out[..., k_b.shape[1]:] = 0.0
    return out


def _absorb_untransposed(q, k_b, d_nope):  # k_b[h]^T applied: sums over the latent index
    qd = core.widen(q)
    lat = np.einsum("hcn,bhc->bhn", core.widen(k_b)[:, :d_nope, :], qd[..., :d_nope])
    pad = np.zeros(qd.shape[:2] + (k_b.shape[1] - d_nope,))
    return np.concatenate([lat, pad, qd[..., d_nope:]], axis=-1)


def _latent_value_from_tail(q_abs, latent, seq_lens, d_c, scale, nthreads=0):
    latent = np.asarray(latent)
    k = np.ascontiguousarray(latent[:, None])
    v = np.ascontiguousarray(latent[:, None, :, -d_c:])
    return core.decode_contig(q_abs, k, v, seq_lens, scale, nthreads)


def _latent_rope_ignored(q_abs, latent, seq_lens, d_c, scale, nthreads=0):
    latent = np.asarray(latent)
    q = np.ascontiguousarray(np.asarray(q_abs)[..., :d_c])
    k = np.ascontiguousarray(latent[:, None, :, :d_c])
    return core.decode_contig(q, k, k, seq_lens, scale, nthreads)


def _unabsorb_transposed(out_lat, v_b):
    vb = core.widen(v_b)
    return np.einsum("hvc,bhv->bhc", vb, core.widen(out_lat)[..., :vb.shape[1]])[..., :vb.shape[1]]


MLA_MUTANTS = [
    ("absorb: rope slice dropped", "mla_absorb_q", _absorb_rope_dropped),
    ("absorb: k_b transposed", "mla_absorb_q", _absorb_untransposed),
    ("latent: value from the row's tail", "decode_mla_absorbed", _latent_value_from_tail),
    ("latent: rope columns ignored", "decode_mla_absorbed", _latent_rope_ignored),
    ("unabsorb: v_b transposed", "mla_unabsorb_out", _unabsorb_transposed),
]


@pytest.mark.parametrize("name,attr,fn", MLA_MUTANTS, ids=[m[0] for m in MLA_MUTANTS])
def test_mla_mutant_is_caught(name, attr, fn):
    core.bind()
    shim = types.SimpleNamespace(**{k: getattr(core, k) for k in dir(core) if not k.startswith("__")})
    setattr(shim, attr, fn)
    failed = []
    for pin in (pins.pin_mla_absorbed_equals_naive, pins.pin_mla_latent_closed_forms, pins.pin_mla_projections):
        try:
            pin(shim)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake '{name}' passed every absorbed-MLA pin"
