"""ctypes binding of the fp64 C oracle (``gqa_oracle.c``).

TEST INFRASTRUCTURE: see the package docstring. Arrays are numpy; bf16 data is
passed as its raw ``uint16`` bit pattern, f32 as ``float32``, f64 as
``float64``. Every function returns fp64 results (or updates buffers of their
own storage type in place, rounding to nearest-even on store).
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16, F64 = 0, 1, 2
_ERRORS = {1: "bad argument", 2: "index out of range", 3: "out of memory"}

_lib = None
_lib_path = None


def bind(path=None):
    """Load the oracle library (the built one by default) and return it."""
    global _lib, _lib_path
    path = path or _build.build()
    l = ctypes.CDLL(path)
    _declare(l)
    _lib, _lib_path = l, path
    return l


def lib():
    if _lib is None:
        bind()
    return _lib


def _declare(_lib):
    if True:
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        _lib.oracle_prefill_causal.argtypes = [P, P, P, P, I, I, I, P, I, I, I, I, D, I, I]
        _lib.oracle_decode_contig.argtypes = [P, P, P, P, P, I, I, I, I, I, I, D, I, I]
        _lib.oracle_decode_paged.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, I, I]
        _lib.oracle_rope_interleaved.argtypes = [P, P, I, I, I, I, I, I, D, I]
        _lib.oracle_kv_append_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, I,
                                                I, I]
        _lib.oracle_attention_arms.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, D, I, D, P, P, I, I]
        _lib.orc_double_to_bf16_bits.argtypes = [D]
        _lib.orc_double_to_bf16_bits.restype = ctypes.c_uint16
        _lib.orc_bf16_bits_to_double.argtypes = [ctypes.c_uint16]
        _lib.orc_bf16_bits_to_double.restype = D
        for f in ("oracle_prefill_causal", "oracle_decode_contig", "oracle_decode_paged",
                  "oracle_rope_interleaved", "oracle_kv_append_paged", "orc_max_threads",
                  "oracle_attention_arms"):
            getattr(_lib, f).restype = ctypes.c_int


def threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return lib().orc_max_threads()


def _et(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle takes float32, bf16 bits (uint16) or float64, got {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    if a is None:
        return None
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))


def _check(rc):
    if rc != 0:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")


def _same_et(*arrs):
    ets = {_et(a) for a in arrs}
    if len(ets) != 1:
        raise TypeError("q, k and v must share one storage type")
    return ets.pop()


def prefill_causal(q, k, v, scale, offsets=None, nthreads=0):
    """q [B, seq_q, H, dk], k [B, Hkv, seq_kv_max, dk], v [B, Hkv, seq_kv_max, dv].
    Row i of batch b sees keys 0..=offsets[b]+i. Returns f64 [B, seq_q, H, dv]."""
    q, k, v = _c(q), _c(k), _c(v)
    B, seq_q, H, dk = q.shape
    _, Hkv, skv, dv = v.shape
    et = _same_et(q, k, v)
    off = None if offsets is None else _c(np.asarray(offsets), np.int32)
    out = np.empty((B, seq_q, H, dv), np.float64)
    _check(lib().oracle_prefill_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, seq_q, skv, _ptr(off),
                                       H, Hkv, dk, dv, float(scale), et, nthreads))
    return out


def decode_contig(q, k, v, seq_lens, scale, nthreads=0):
    """q [B, H, dk], k [B, Hkv, max_len, dk], v [B, Hkv, max_len, dv]; seq_lens[b]
    counts rows present including the query's own. Returns f64 [B, H, dv]."""
    q, k, v = _c(q), _c(k), _c(v)
    B, H, dk = q.shape
    _, Hkv, max_len, dv = v.shape
    et = _same_et(q, k, v)
    lens = _c(np.asarray(seq_lens), np.int32)
    out = np.empty((B, H, dv), np.float64)
    _check(lib().oracle_decode_contig(_ptr(q), _ptr(k), _ptr(v), _ptr(lens), _ptr(out), B, max_len, H,
                                      Hkv, dk, dv, float(scale), et, nthreads))
    return out


def attention_arms(q, k, v, base_len, scale, window=0, softcap=0.0, sinks=None, slopes=None, nthreads=0):
    """Query rows with the arms (gqa_oracle.c, `oracle_attention_arms`):
    q [B, seq_q, H, dk] (or [B, H, dk] for one row), k [B, Hkv, max_len, dk],
    v [B, Hkv, max_len, dv]; base_len[b] = keys present after this pass's rows
    (row i sits at position base_len[b] - seq_q + i). window <= 0 and softcap
    <= 0 switch those arms off; sinks and slopes are [H] or None. Returns f64
    with q's leading shape and d_v last."""
    q, k, v = _c(q), _c(k), _c(v)
    one_row = q.ndim == 3
    q4 = q.reshape(q.shape[0], 1, q.shape[1], q.shape[2]) if one_row else q
    B, seq_q, H, dk = q4.shape
    _, Hkv, max_len, dv = v.shape
    et = _same_et(q4, k, v)
    base = _c(np.asarray(base_len), np.int32)
    sk = None if sinks is None else _c(np.asarray(sinks, np.float64), np.float64)
    sl = None if slopes is None else _c(np.asarray(slopes, np.float64), np.float64)
    out = np.empty((B, seq_q, H, dv), np.float64)
    _check(lib().oracle_attention_arms(_ptr(q4), _ptr(k), _ptr(v), _ptr(base), _ptr(out), B, seq_q, max_len, H,
                                       Hkv, dk, dv, float(scale), int(window), float(softcap),
                                       None if sk is None else _ptr(sk), None if sl is None else _ptr(sl), et,
                                       nthreads))
    return out.reshape(B, H, dv) if one_row else out


def decode_paged(q, k_pool, v_pool, tables, seq_lens, scale, nthreads=0):
    """q [B, H, dk]; pools [num_blocks, Hkv, bs, d]; tables int32 [B, mbps]."""
    q, k_pool, v_pool = _c(q), _c(k_pool), _c(v_pool)
    B, H, dk = q.shape
    nb, Hkv, bs, dv = v_pool.shape
    et = _same_et(q, k_pool, v_pool)
    tables = _c(np.asarray(tables), np.int32)
    lens = _c(np.asarray(seq_lens), np.int32)
    out = np.empty((B, H, dv), np.float64)
    _check(lib().oracle_decode_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(tables), _ptr(lens),
                                     _ptr(out), B, tables.shape[1], nb, bs, H, Hkv, dk, dv,
                                     float(scale), et, nthreads))
    return out


def decode_mla_naive(q, k_nope, k_rot, v, seq_lens, scale, nthreads=0):
    """MLA-shaped decode in the naive per-head form of frink-models src/mla/mod.rs
    (`naive_attention`): every head's key row is concat(k_nope[b,h,j], k_rot[b,j]),
    the shared rotated vector copied into each head. The copy is materialised here
    (group size 1: KV head = query head). q [B, H, dn+dr], k_nope [B, H, L, dn],
    k_rot [B, L, dr], v [B, H, L, dv]."""
    B, H, L, dn = k_nope.shape
    dr = k_rot.shape[-1]
    k_full = np.empty((B, H, L, dn + dr), k_nope.dtype)
    k_full[..., :dn] = k_nope
    k_full[..., dn:] = k_rot[:, None, :, :]
    return decode_contig(q, k_full, v, seq_lens, scale, nthreads)


def mla_absorb_q(q, k_b, d_nope):
    """Absorbed query of frink-models src/mla/mod.rs (`absorbed_attention`, the
    `MlaKvB::Split` form): for every head, the nope slice q[b, h, :d_nope] is
    mapped into the latent space by k_b[h] ([d_c, d_nope], the absorb direction),
    and the rope slice q[b, h, d_nope:] is kept as it is. q [B, H, d_nope + d_r],
    k_b [H, d_c, d_nope]. Returns f64 [B, H, d_c + d_r]."""
    qd, kb = widen(np.asarray(q)), widen(np.asarray(k_b))
    absorbed = np.einsum("hcn,bhn->bhc", kb, qd[..., :d_nope])
    return np.concatenate([absorbed, qd[..., d_nope:]], axis=-1)


def decode_mla_absorbed(q_abs, latent, seq_lens, d_c, scale, nthreads=0):
    """Attention over the latent cache (frink-models src/mla/mod.rs,
    `absorbed_attention`: MQA over rows of width kv_lora_rank + qk_rope, every
    head attending to the same row). Row j of sequence b is latent[b, j] =
    (c_j, k_rot_j); its key is the whole row and its value the first d_c
    columns, c_j. q_abs [B, H, d_c + d_r], latent [B, max_len, d_c + d_r], both of
    one storage type; seq_lens[b] rows are visible. Returns f64 [B, H, d_c]."""
    latent = np.asarray(latent)
    k = np.ascontiguousarray(latent[:, None, :, :])
    v = np.ascontiguousarray(latent[:, None, :, :d_c])
    return decode_contig(q_abs, k, v, seq_lens, scale, nthreads)


def mla_unabsorb_out(out_lat, v_b):
    """Output of the absorbed form (frink-models src/mla/mod.rs,
    `absorbed_attention`): each head's weighted latent out_lat[b, h] ([d_c]) is
    mapped to the value width by v_b[h] ([d_v, d_c]). Returns f64 [B, H, d_v]."""
    return np.einsum("hvc,bhc->bhv", widen(np.asarray(v_b)), widen(np.asarray(out_lat)))


def rope_interleaved(x, positions, rot_offset, rot_dim, theta):
    """Interleaved RoPE of x [B, T, heads, d] at positions [B, T]; returns a new
    array of x's storage type (f32/bf16 results rounded to nearest-even)."""
    x = np.array(x, copy=True, order="C")
    B, T, heads, d = x.shape
    pos = _c(np.asarray(positions).reshape(B, T), np.int32)
    _check(lib().oracle_rope_interleaved(_ptr(x), _ptr(pos), B, T, heads, d, rot_offset, rot_dim,
                                         float(theta), _et(x)))
    return x


def kv_append_paged(q, k_new, v_new, k_pool, v_pool, tables, seq_lens_in, theta, rot_offset=0,
                    rot_dim=None):
    """Returns (q_rotated, k_pool', v_pool', seq_lens_out) as new arrays."""
    q = np.array(q, copy=True, order="C")
    k_pool = np.array(k_pool, copy=True, order="C")
    v_pool = np.array(v_pool, copy=True, order="C")
    k_new, v_new = _c(k_new), _c(v_new)
    B, H, dk = q.shape
    nb, Hkv, bs, dv = v_pool.shape
    et = _same_et(q, k_new, v_new, k_pool, v_pool)
    tables = _c(np.asarray(tables), np.int32)
    lin = _c(np.asarray(seq_lens_in), np.int32)
    lout = np.empty_like(lin)
    rot_dim = dk - rot_offset if rot_dim is None else rot_dim
    _check(lib().oracle_kv_append_paged(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                        _ptr(tables), _ptr(lin), _ptr(lout), B, tables.shape[1], nb, bs,
                                        H, Hkv, dk, dv, float(theta), rot_offset, rot_dim, et))
    return q, k_pool, v_pool, lout


def bf16_bits(x: float) -> int:
    """The oracle's own nearest-even rounding of a double to a bf16 bit pattern."""
    return int(lib().orc_double_to_bf16_bits(float(x)))


def bf16_value(bits: int) -> float:
    return float(lib().orc_bf16_bits_to_double(int(bits)))


def widen(a: np.ndarray) -> np.ndarray:
    """Exact widening of f32 / bf16-bits / f64 storage to float64."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


if os.environ.get("ORACLE_BUILD_ON_IMPORT"):
    lib()
