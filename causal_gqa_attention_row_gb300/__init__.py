"""Python binding of libgqa_attn.so (include/gqa_attn.h).

Argument marshalling only: every function here takes torch tensors that already
live on the GPU, checks their dtype, shape and contiguity, and passes raw
pointers, sizes and the current CUDA stream to the C entry point of the same
name. All arithmetic runs in the library's CUDA kernels; there is no fallback.
If the shared library is missing, ``load()`` raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_attn.so")

F32, BF16 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "CUDA error",
          4: "workspace missing or too small", 5: "device saw an index or length out of range",
          6: "a bounded device wait gave up"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_DEVICE_BOUNDS, ERR_DEVICE_TIMEOUT = range(7)

EXPORTS = ("attn_prefill_causal", "attn_decode_contig", "attn_decode_paged", "kv_append_paged",
           "attn_rope_interleaved", "attn_decode_workspace_bytes", "attn_get_device_error",
           "gqa_status_string", "gqa_debug_withhold_first_tile", "attn_decode_paged_static_workspace",
           "attn_prefill_causal_ex", "attn_decode_contig_ex", "attn_decode_paged_ex", "attn_prefill_paged",
           "attn_prefill_paged_ex", "mla_absorb_q", "attn_decode_mla_absorbed",
           "attn_decode_mla_absorbed_workspace_bytes", "mla_unabsorb_out", "attn_decode_mla_absorbed_paged",
           "attn_rope_interleaved_qk")


class GqaArms(ctypes.Structure):
    """`gqa_arms` (include/gqa_attn.h): window, softcap, sinks, ALiBi slopes."""
    _fields_ = [("window", ctypes.c_int), ("softcap", ctypes.c_float), ("sinks", ctypes.c_void_p),
                ("alibi_slopes", ctypes.c_void_p)]

STATIC_WORKSPACE_BYTES = 16 << 20  # GQA_STATIC_WORKSPACE_BYTES

_lib = None


class GqaError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status})")


def load(path: str = None):
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, F, D, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t
    sig = {
        "attn_prefill_causal": [P, P, P, P, I, I, I, P, I, I, I, I, F, I, P],
        "attn_decode_contig": [P, P, P, P, I, P, P, I, I, I, I, I, I, F, I, P, S, P],
        "attn_decode_paged": [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P, S, P],
        "attn_decode_paged_static_workspace": [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P],
        "kv_append_paged": [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, I, I, I, P],
        "attn_rope_interleaved": [P, P, I, I, I, I, I, I, I, D, I, P],
        "attn_rope_interleaved_qk": [P, P, P, I, I, I, I, I, I, I, I, I, D, I, P],
        "attn_get_device_error": [P],
        "attn_prefill_causal_ex": [P, P, P, P, I, I, I, P, I, I, I, I, F, I, P, P],
        "attn_decode_contig_ex": [P, P, P, P, I, P, P, I, I, I, I, I, I, F, I, P, S, P, P],
        "attn_decode_paged_ex": [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P, S, P, P],
        "attn_prefill_paged": [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P],
        "attn_prefill_paged_ex": [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P, P],
        "gqa_debug_withhold_first_tile": [I],
        "mla_absorb_q": [P, P, P, I, I, I, I, I, I, P],
        "attn_decode_mla_absorbed": [P, P, P, P, I, I, I, I, I, F, I, P, S, P],
        "mla_unabsorb_out": [P, P, P, I, I, I, I, I, P],
        "attn_decode_mla_absorbed_paged": [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, S, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.attn_decode_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_decode_workspace_bytes.restype = S
    lib.attn_decode_mla_absorbed_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_decode_mla_absorbed_workspace_bytes.restype = S
    lib.gqa_status_string.argtypes = [I]
    lib.gqa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _dtype(*ts):
    dts = {t.dtype for t in ts if t is not None}
    if len(dts) != 1:
        raise TypeError(f"tensors must share one dtype, got {dts}")
    dt = dts.pop()
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {dt}")


def _p(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _i32(t):
    if t is not None and t.dtype != torch.int32:
        raise TypeError("index tensors must be int32")
    return _p(t)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, what):
    if status != OK:
        raise GqaError(status, what)


def _arms(window, softcap, sinks, alibi_slopes):
    """The `gqa_arms` struct (by reference), or None when every arm is off."""
    if not window and not softcap and sinks is None and alibi_slopes is None:
        return None
    for t in (sinks, alibi_slopes):
        if t is not None and t.dtype != torch.float32:
            raise TypeError("sinks and alibi_slopes must be float32 [H]")
    return ctypes.byref(GqaArms(int(window or 0), float(softcap or 0.0), _p(sinks), _p(alibi_slopes)))


def attn_prefill_causal(q, k, v, out, attention_scale, position_offset=None, stream=None, window=0, softcap=0.0,
                        sinks=None, alibi_slopes=None):
    """q [B, S, H, dk], k [B, Hkv, S_kv, dk], v [B, Hkv, S_kv, dv], out [B, S, H, dv].
    window / softcap / sinks / alibi_slopes: the arms (include/gqa_attn.h, `gqa_arms`)."""
    B, S, H, dk = q.shape
    _, Hkv, S_kv, dv = v.shape
    arms = _arms(window, softcap, sinks, alibi_slopes)
    args = (_p(q), _p(k), _p(v), _p(out), B, S, S_kv, _i32(position_offset), H, Hkv, dk, dv, float(attention_scale),
            _dtype(q, k, v, out))
    if arms is None:
        _check(load().attn_prefill_causal(*args, _stream(stream)), "attn_prefill_causal")
    else:
        _check(load().attn_prefill_causal_ex(*args, arms, _stream(stream)), "attn_prefill_causal_ex")
    return out


def attn_prefill_paged(q, k_pool, v_pool, block_tables, out, attention_scale, position_offset=None, stream=None,
                       window=0, softcap=0.0, sinks=None, alibi_slopes=None):
    """Chunked prefill against the paged pool: q [B, S, H, dk]; pools [num_blocks, Hkv, bs, d];
    block_tables int32 [B, mbps]; position_offset int32 [B] or None; out [B, S, H, dv].
    window / softcap / sinks / alibi_slopes: the arms (`gqa_arms`)."""
    B, S, H, dk = q.shape
    nb, Hkv, bs, dv = v_pool.shape
    arms = _arms(window, softcap, sinks, alibi_slopes)
    args = (_p(q), _p(k_pool), _p(v_pool), _i32(block_tables), _i32(position_offset), _p(out), B, S,
            block_tables.shape[1], nb, bs, H, Hkv, dk, dv, float(attention_scale), _dtype(q, k_pool, v_pool, out))
    if arms is None:
        _check(load().attn_prefill_paged(*args, _stream(stream)), "attn_prefill_paged")
    else:
        _check(load().attn_prefill_paged_ex(*args, arms, _stream(stream)), "attn_prefill_paged_ex")
    return out


def attn_decode_workspace_bytes(B, H, d_v, max_len):
    return int(load().attn_decode_workspace_bytes(B, H, d_v, max_len))


def decode_workspace(B, H, d_v, max_len, device="cuda"):
    """A workspace tensor of the size the decode calls need (None when none)."""
    n = attn_decode_workspace_bytes(B, H, d_v, max_len)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def attn_decode_contig(q, k_cache, v_cache, seq_lens, out, attention_scale, workspace=None, k_rot_shared=None,
                       stream=None, window=0, softcap=0.0, sinks=None, alibi_slopes=None):
    """q [B, H, dk]; k_cache [B, Hkv, L, dk - d_rot]; v_cache [B, Hkv, L, dv];
    k_rot_shared None or [B, L, d_rot]; seq_lens int32 [B]; out [B, H, dv];
    window / softcap / sinks / alibi_slopes: the arms (`gqa_arms`)."""
    B, H, dk = q.shape
    _, Hkv, L, dv = v_cache.shape
    d_rot = 0 if k_rot_shared is None else k_rot_shared.shape[-1]
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    arms = _arms(window, softcap, sinks, alibi_slopes)
    args = (_p(q), _p(k_cache), _p(v_cache), _p(k_rot_shared), d_rot, _i32(seq_lens), _p(out), B, L, H, Hkv, dk, dv,
            float(attention_scale), _dtype(q, k_cache, v_cache, out, k_rot_shared), _p(workspace), ws)
    if arms is None:
        _check(load().attn_decode_contig(*args, _stream(stream)), "attn_decode_contig")
    else:
        _check(load().attn_decode_contig_ex(*args, arms, _stream(stream)), "attn_decode_contig_ex")
    return out


def attn_decode_paged(q, k_pool, v_pool, block_tables, seq_lens, out, attention_scale, workspace=None,
                      stream=None, window=0, softcap=0.0, sinks=None, alibi_slopes=None):
    """q [B, H, dk]; pools [num_blocks, Hkv, bs, d]; block_tables int32 [B, mbps];
    window / softcap / sinks / alibi_slopes: the arms (`gqa_arms`)."""
    B, H, dk = q.shape
    nb, Hkv, bs, dv = v_pool.shape
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    arms = _arms(window, softcap, sinks, alibi_slopes)
    args = (_p(q), _p(k_pool), _p(v_pool), _i32(block_tables), _i32(seq_lens), _p(out), B, block_tables.shape[1], nb,
            bs, H, Hkv, dk, dv, float(attention_scale), _dtype(q, k_pool, v_pool, out), _p(workspace), ws)
    if arms is None:
        _check(load().attn_decode_paged(*args, _stream(stream)), "attn_decode_paged")
    else:
        _check(load().attn_decode_paged_ex(*args, arms, _stream(stream)), "attn_decode_paged_ex")
    return out


def attn_decode_paged_static_workspace(q, k_pool, v_pool, block_tables, seq_lens, out, attention_scale,
                                       stream=None):
    """attn_decode_paged with the library's fixed device scratch instead of a
    caller-allocated workspace (for callers that cannot allocate device memory;
    see include/gqa_attn.h). Raises GqaError(ERR_WORKSPACE) when the problem needs
    more than STATIC_WORKSPACE_BYTES of scratch."""
    B, H, dk = q.shape
    nb, Hkv, bs, dv = v_pool.shape
    _check(load().attn_decode_paged_static_workspace(_p(q), _p(k_pool), _p(v_pool), _i32(block_tables),
                                                     _i32(seq_lens), _p(out), B, block_tables.shape[1], nb, bs, H,
                                                     Hkv, dk, dv, float(attention_scale),
                                                     _dtype(q, k_pool, v_pool, out), _stream(stream)),
           "attn_decode_paged_static_workspace")
    return out


def mla_absorb_q(q, k_b, q_abs, stream=None):
    """q [B, H, d_nope + d_rope]; k_b [H, d_c, d_nope]; q_abs [B, H, d_c + d_rope] (bf16)."""
    B, H, dq = q.shape
    _, d_c, d_nope = k_b.shape
    _check(load().mla_absorb_q(_p(q), _p(k_b), _p(q_abs), B, H, d_nope, dq - d_nope, d_c, _dtype(q, k_b, q_abs),
                               _stream(stream)), "mla_absorb_q")
    return q_abs


def attn_decode_mla_absorbed_workspace_bytes(B, H, d_c, max_len):
    return int(load().attn_decode_mla_absorbed_workspace_bytes(B, H, d_c, max_len))


def mla_absorbed_workspace(B, H, d_c, max_len, device="cuda"):
    """A workspace tensor of the size attn_decode_mla_absorbed needs (None when none)."""
    n = attn_decode_mla_absorbed_workspace_bytes(B, H, d_c, max_len)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def attn_decode_mla_absorbed(q_abs, latent, seq_lens, out_lat, attention_scale, workspace=None, stream=None):
    """q_abs [B, H, d_c + d_r]; latent [B, L, d_c + d_r]; seq_lens int32 [B];
    out_lat [B, H, d_c] (bf16)."""
    B, H, w = q_abs.shape
    _, L, _ = latent.shape
    d_c = out_lat.shape[-1]
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().attn_decode_mla_absorbed(_p(q_abs), _p(latent), _i32(seq_lens), _p(out_lat), B, L, H, d_c, w - d_c,
                                           float(attention_scale), _dtype(q_abs, latent, out_lat), _p(workspace), ws,
                                           _stream(stream)), "attn_decode_mla_absorbed")
    return out_lat


def attn_decode_mla_absorbed_paged(q_abs, latent_pool, block_tables, seq_lens, out_lat, attention_scale,
                                   workspace=None, stream=None):
    """q_abs [B, H, d_c + d_r]; latent_pool [num_blocks, bs, d_c + d_r]; block_tables int32
    [B, mbps]; seq_lens int32 [B]; out_lat [B, H, d_c] (bf16)."""
    B, H, w = q_abs.shape
    nb, bs, _ = latent_pool.shape
    d_c = out_lat.shape[-1]
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().attn_decode_mla_absorbed_paged(_p(q_abs), _p(latent_pool), _i32(block_tables), _i32(seq_lens),
                                                 _p(out_lat), B, block_tables.shape[1], nb, bs, H, d_c, w - d_c,
                                                 float(attention_scale), _dtype(q_abs, latent_pool, out_lat),
                                                 _p(workspace), ws, _stream(stream)),
           "attn_decode_mla_absorbed_paged")
    return out_lat


def mla_unabsorb_out(out_lat, v_b, out, stream=None):
    """out_lat [B, H, d_c]; v_b [H, d_v, d_c]; out [B, H, d_v] (bf16)."""
    B, H, d_c = out_lat.shape
    d_v = v_b.shape[1]
    _check(load().mla_unabsorb_out(_p(out_lat), _p(v_b), _p(out), B, H, d_c, d_v, _dtype(out_lat, v_b, out),
                                   _stream(stream)), "mla_unabsorb_out")
    return out


def kv_append_paged(q, k_new, v_new, k_pool, v_pool, block_tables, seq_lens_in, seq_lens_out, rope_theta,
                    rot_offset=0, rot_dim=None, stream=None):
    """Rotate q and k_new at p = seq_lens_in[b], write k/v into the pools, set
    seq_lens_out = p + 1 (may be the same tensor as seq_lens_in)."""
    B, H, dk = q.shape
    nb, Hkv, bs, dv = v_pool.shape
    rot_dim = dk - rot_offset if rot_dim is None else rot_dim
    _check(load().kv_append_paged(_p(q), _p(k_new), _p(v_new), _p(k_pool), _p(v_pool), _i32(block_tables),
                                  _i32(seq_lens_in), _i32(seq_lens_out), B, block_tables.shape[1], nb, bs, H,
                                  Hkv, dk, dv, float(rope_theta), rot_offset, rot_dim,
                                  _dtype(q, k_new, v_new, k_pool, v_pool), _stream(stream)), "kv_append_paged")


def attn_rope_interleaved(x, positions, theta, rot_offset=0, rot_dim=None, heads_outer=False, stream=None):
    """In place. x [B, T, heads, d] (or [B, heads, T, d] with heads_outer); positions int32 [B, T]."""
    if heads_outer:
        B, heads, T, d = x.shape
    else:
        B, T, heads, d = x.shape
    rot_dim = d - rot_offset if rot_dim is None else rot_dim
    _check(load().attn_rope_interleaved(_p(x), _i32(positions), B, T, heads, d, int(bool(heads_outer)),
                                        rot_offset, rot_dim, float(theta), _dtype(x), _stream(stream)),
           "attn_rope_interleaved")
    return x


def attn_rope_interleaved_qk(q, k, positions, theta, rot_offset=0, rot_dim=None, q_heads_outer=False,
                             k_heads_outer=False, stream=None):
    """In place, one launch. q [B, T, heads_q, d] (or [B, heads_q, T, d] with
    q_heads_outer), k likewise; positions int32 [B, T]."""
    if q_heads_outer:
        B, hq, T, d = q.shape
    else:
        B, T, hq, d = q.shape
    hk = k.shape[1] if k_heads_outer else k.shape[2]
    rot_dim = d - rot_offset if rot_dim is None else rot_dim
    _check(load().attn_rope_interleaved_qk(_p(q), _p(k), _i32(positions), B, T, hq, hk, d, int(bool(q_heads_outer)),
                                           int(bool(k_heads_outer)), rot_offset, rot_dim, float(theta), _dtype(q),
                                           _stream(stream)), "attn_rope_interleaved_qk")
    return q, k


def attn_get_device_error(stream=None):
    """Synchronise the stream; return (and clear) the device error status code."""
    return int(load().attn_get_device_error(_stream(stream)))


def gqa_status_string(status):
    return load().gqa_status_string(int(status)).decode()


def gqa_debug_withhold_first_tile(enable):
    return int(load().gqa_debug_withhold_first_tile(int(bool(enable))))
