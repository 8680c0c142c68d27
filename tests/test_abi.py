"""The C ABI library (CPU only): it loads, exports every symbol include/gqa_attn.h
declares, and rejects host-checkable bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from causal_gqa_attention_row_gb300 import build
    build.build()
    import causal_gqa_attention_row_gb300 as g
    return g.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gqa_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"if", "sizeof"}


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"attn_prefill_causal", "attn_decode_contig", "attn_decode_paged", "kv_append_paged",
            "attn_rope_interleaved", "attn_decode_workspace_bytes", "attn_get_device_error"} <= names
    for n in names:
        assert hasattr(lib, n), n
    import causal_gqa_attention_row_gb300 as g
    assert names <= set(g.EXPORTS)


def test_status_strings(lib):
    import causal_gqa_attention_row_gb300 as g
    for s in range(7):
        assert g.gqa_status_string(s) == g.STATUS[s]


def test_workspace_size(lib):
    import causal_gqa_attention_row_gb300 as g
    assert g.attn_decode_workspace_bytes(256, 32, 128, 2048) == 0          # one split: none needed
    units = 256 * 32 * 17                       # (sequence, head, split) slots, 2048-row splits
    plan = 256 + (units * 8 + 255) // 256 * 256  # ticket header + split list
    assert g.attn_decode_workspace_bytes(256, 32, 128, 2049 * 16) == plan + units * 130 * 4
    assert g.attn_decode_workspace_bytes(0, 32, 128, 5000) == 0


def test_bad_arguments_rejected_before_launch(lib):
    """Each call below fails a host check, so it returns before any CUDA call."""
    P = ctypes.c_void_p(16)  # a non-null, 16-byte aligned stand-in: never dereferenced
    N = None
    inv = 1
    # H % Hkv != 0
    assert lib.attn_decode_contig(P, P, P, N, 0, P, P, 2, 64, 6, 4, 128, 128, 0.1, 1, N, 0, N) == inv
    # d_k not a multiple of 8
    assert lib.attn_decode_paged(P, P, P, P, P, P, 2, 4, 10, 16, 8, 2, 100, 100, 0.1, 1, N, 0, N) == inv
    # null q
    assert lib.attn_decode_paged(N, P, P, P, P, P, 2, 4, 10, 16, 8, 2, 128, 128, 0.1, 1, N, 0, N) == inv
    # unknown dtype
    assert lib.attn_prefill_causal(P, P, P, P, 1, 8, 8, N, 4, 2, 16, 16, 0.25, 7, N) == inv
    # seq_q > seq_kv_max
    assert lib.attn_prefill_causal(P, P, P, P, 1, 9, 8, N, 4, 2, 16, 16, 0.25, 0, N) == inv
    # k_rot given without d_rot
    assert lib.attn_decode_contig(P, P, P, P, 0, P, P, 2, 64, 8, 8, 192, 128, 0.1, 1, N, 0, N) == inv
    # misaligned pointer
    assert lib.attn_decode_contig(ctypes.c_void_p(18), P, P, N, 0, P, P, 2, 64, 8, 8, 128, 128, 0.1, 1, N, 0,
                                  N) == inv
    # odd rot_dim, theta <= 0
    assert lib.attn_rope_interleaved(P, P, 1, 4, 2, 64, 0, 0, 63, 1e4, 1, N) == inv
    assert lib.attn_rope_interleaved(P, P, 1, 4, 2, 64, 0, 0, 64, 0.0, 1, N) == inv
    # rotated slice past the head
    assert lib.kv_append_paged(P, P, P, P, P, P, P, P, 2, 4, 10, 16, 8, 2, 64, 64, 1e4, 16, 64, 1, N) == inv
    # the arms: a softcap that is not finite, a misaligned sink array
    import causal_gqa_attention_row_gb300 as g
    nan_cap = g.GqaArms(0, float("nan"), None, None)
    assert lib.attn_decode_contig_ex(P, P, P, N, 0, P, P, 2, 64, 8, 2, 128, 128, 0.1, 1, N, 0,
                                     ctypes.byref(nan_cap), N) == inv
    bad_sinks = g.GqaArms(16, 0.0, 18, None)
    assert lib.attn_decode_paged_ex(P, P, P, P, P, P, 2, 4, 10, 16, 8, 2, 128, 128, 0.1, 1, N, 0,
                                    ctypes.byref(bad_sinks), N) == inv
    # empty batches are no-ops
    assert lib.attn_decode_contig(N, N, N, N, 0, N, N, 0, 64, 8, 2, 128, 128, 0.1, 1, N, 0, N) == 0


def test_mla_absorbed_workspace_and_checks(lib):
    """The absorbed-MLA calls: workspace size and host-side rejections (no launch)."""
    import causal_gqa_attention_row_gb300 as g
    # splits of C rows: C = 1024, doubled while B * ceil(H / 128) * ceil(max_len / 2C) >= 64
    assert g.attn_decode_mla_absorbed_workspace_bytes(32, 128, 512, 1024) == 0   # one split: none
    assert g.attn_decode_mla_absorbed_workspace_bytes(32, 128, 512, 4096) == 32 * 128 * 2 * 514 * 4  # C = 2048
    assert g.attn_decode_mla_absorbed_workspace_bytes(32, 128, 512, 1500) == 32 * 128 * 2 * 514 * 4  # C = 1024
    assert g.attn_decode_mla_absorbed_workspace_bytes(2, 16, 512, 1025) == 2 * 16 * 2 * 514 * 4      # C = 1024
    assert g.attn_decode_mla_absorbed_workspace_bytes(64, 256, 512, 32768) == 64 * 256 * 4 * 514 * 4  # C = 8192
    assert g.attn_decode_mla_absorbed_workspace_bytes(1, 128, 512, 32768) == 1 * 128 * 32 * 514 * 4  # C = 1024
    P = ctypes.c_void_p(16)
    N = None
    # (q_abs, latent, seq_lens, out_lat, B, max_len, H, d_c, d_r, scale, dtype, workspace, bytes, stream)
    assert lib.attn_decode_mla_absorbed(P, P, P, P, 2, 64, 16, 256, 64, 0.07, 1, N, 0, N) == 2   # widths
    assert lib.attn_decode_mla_absorbed(P, P, P, P, 2, 64, 16, 512, 64, 0.07, 0, N, 0, N) == 2   # f32
    assert lib.attn_decode_mla_absorbed(P, P, P, P, 2, 64, 16, 512, 64, 0.0, 1, N, 0, N) == 2    # scale
    assert lib.attn_decode_mla_absorbed(N, P, P, P, 2, 64, 16, 512, 64, 0.07, 1, N, 0, N) == 1   # null
    assert lib.attn_decode_mla_absorbed(ctypes.c_void_p(24), P, P, P, 2, 64, 16, 512, 64, 0.07, 1, N, 0,
                                        N) == 1                                                   # misaligned
    assert lib.attn_decode_mla_absorbed(P, P, P, P, 2, 4096, 16, 512, 64, 0.07, 1, N, 0, N) == 4  # workspace
    assert lib.attn_decode_mla_absorbed(N, N, N, N, 0, 64, 16, 512, 64, 0.07, 1, N, 0, N) == 0    # empty batch
    # (q, k_b, q_abs, B, H, d_nope, d_rope, d_c, dtype, stream)
    assert lib.mla_absorb_q(P, P, P, 2, 16, 128, 64, 512, 1, N) == 1                              # q_abs aliases q
    assert lib.mla_absorb_q(P, P, ctypes.c_void_p(32), 2, 16, 128, 64, 512, 0, N) == 2            # f32
    # (out_lat, v_b, out, B, H, d_c, d_v, dtype, stream)
    assert lib.mla_unabsorb_out(P, P, P, 2, 16, 512, 128, 1, N) == 1                              # aliasing
    assert lib.mla_unabsorb_out(P, P, ctypes.c_void_p(32), 2, 16, 0, 128, 1, N) == 1              # d_c


def test_mla_absorbed_paged_checks(lib):
    P = ctypes.c_void_p(16)
    N = None
    # (q_abs, pool, tables, seq_lens, out, B, mbps, num_blocks, bs, H, d_c, d_r, scale, dtype, ws, bytes, stream)
    assert lib.attn_decode_mla_absorbed_paged(P, P, P, P, P, 2, 8, 100, 24, 16, 512, 64, 0.07, 1, N, 0, N) == 2
    assert lib.attn_decode_mla_absorbed_paged(P, P, N, P, P, 2, 8, 100, 16, 16, 512, 64, 0.07, 1, N, 0, N) == 1
    assert lib.attn_decode_mla_absorbed_paged(P, P, P, P, P, 2, 0, 100, 16, 16, 512, 64, 0.07, 1, N, 0, N) == 1
    assert lib.attn_decode_mla_absorbed_paged(P, P, P, P, P, 2, 128, 100, 16, 16, 512, 64, 0.07, 1, N, 0,
                                              N) == 4  # 2048 rows: two splits need a workspace
    assert lib.attn_decode_mla_absorbed_paged(N, N, N, N, N, 0, 8, 100, 16, 16, 512, 64, 0.07, 1, N, 0, N) == 0


def test_static_workspace_size_matches_header():
    """The binding's STATIC_WORKSPACE_BYTES is the header's GQA_STATIC_WORKSPACE_BYTES."""
    import causal_gqa_attention_row_gb300 as g
    text = open(os.path.join(ROOT, "include", "gqa_attn.h")).read()
    m = re.search(r"#define\s+GQA_STATIC_WORKSPACE_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "GQA_STATIC_WORKSPACE_BYTES not found in the header"
    assert g.STATIC_WORKSPACE_BYTES == int(m.group(1)) << int(m.group(2))
