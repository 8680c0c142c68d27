"""The seeded input generators (CPU): the same seed gives the same tensors, the
shapes and scales are the documented ones."""
import math

import torch

import workloads as W


def test_absorbed_mla_inputs_are_seeded_and_shaped():
    a = W.make_mla_absorbed(B=2, H=4, max_len=12, lens=[12, 5], seed=3)
    b = W.make_mla_absorbed(B=2, H=4, max_len=12, lens=[12, 5], seed=3)
    for x, y in ((a.q, b.q), (a.k_b, b.k_b), (a.v_b, b.v_b), (a.latent, b.latent)):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    assert a.q.shape == (2, 4, 192) and a.k_b.shape == (4, 512, 128) and a.v_b.shape == (4, 128, 512)
    assert a.latent.shape == (2, 12, 576) and a.lens.tolist() == [12, 5]
    assert abs(a.scale - 1 / math.sqrt(192)) < 1e-15
    # synthetic projections keep unit scale: k_b ~ N(0, 1/128), v_b ~ N(0, 1/512)
    assert abs(a.k_b.float().std().item() * math.sqrt(128) - 1) < 0.05
    assert abs(a.v_b.float().std().item() * math.sqrt(512) - 1) < 0.05
    c = W.make_mla_absorbed(B=2, H=4, max_len=12, seed=4)
    assert not torch.equal(a.latent, c.latent) and c.lens.tolist() == [12, 12]


def test_paged_tables_are_disjoint_and_cover_the_appended_row():
    c = W.make_paged(B=5, H=8, Hkv=2, dk=16, dv=16, block_size=4, num_blocks=300, len_hi=40, seed=7)
    seen = set()
    for b in range(5):
        n = int(c.seq_lens[b]) + 1  # the history and the appended row
        need = (n + 3) // 4
        row = c.tables[b].tolist()
        assert all(e >= 0 for e in row[:need]) and all(e == -1 for e in row[need:])
        assert not (set(row[:need]) & seen)
        seen |= set(row[:need])
