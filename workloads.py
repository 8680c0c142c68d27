"""Seeded synthetic inputs for causal GQA attention against a KV cache.

The one module both the CUDA path's callers and the oracle's callers share. It
holds shapes and random numbers only -- no step of the attention arithmetic,
no RoPE, no indexing rule of the method. Values are N(0, 1) drawn with a seeded
``torch.Generator`` and rounded to the storage dtype by torch (nearest-even).

Workloads (the five of the attention pages' problem statement, at full size):

* tiny fp32  -- H=4, Hkv=2, d=16, 8-row prefill, one decode step, paged bs=4
* prefill    -- batch 1, H=14, Hkv=2, d=64, 2048 rows, RoPE theta 1e6
* contig     -- 64 sequences, H=32, Hkv=8, d=128, cache length U[512, 8192]
* paged      -- 256 sequences, H=32, Hkv=8, d=128, block size 16, a 600,000-block
                pool, block tables from a seeded permutation, history U[1, 32768],
                one appended row per sequence (RoPE theta 1e6)
* mla        -- 32 sequences, 128 heads, group 1, d_k = 128 + 64 (shared k_rot,
                RoPE theta 1e4), d_v = 128, cache length 4096
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, g: torch.Generator, dtype=torch.float32, device="cpu") -> torch.Tensor:
    """N(0,1) of `dtype`; large tensors are filled in chunks (no fp32 staging copy)."""
    t = torch.empty(shape, dtype=dtype, device=device)
    flat = t.view(-1)
    step = 1 << 28
    for s in range(0, flat.numel(), step):
        flat[s:s + step].normal_(generator=g)
    return t


def to_oracle(t: torch.Tensor) -> np.ndarray:
    """Storage view for the oracle: bf16 -> uint16 bit pattern, f32 -> float32."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float32, torch.float64, torch.int32, torch.int64):
        return t.numpy()
    raise TypeError(t.dtype)


@dataclass
class PrefillCase:
    q: torch.Tensor           # [B, S, H, dk]
    k: torch.Tensor           # [B, Hkv, S_kv, dk]
    v: torch.Tensor           # [B, Hkv, S_kv, dv]
    offsets: torch.Tensor     # int32 [B]
    scale: float
    theta: float = 0.0


@dataclass
class ContigCase:
    q: torch.Tensor           # [B, H, dk]
    k: torch.Tensor           # [B, Hkv, max_len, dk - d_rot]
    v: torch.Tensor           # [B, Hkv, max_len, dv]
    seq_lens: torch.Tensor    # int32 [B], rows present including the query's own
    scale: float
    k_rot: torch.Tensor = None  # [B, max_len, d_rot] (MLA-shaped shared rotated part)


@dataclass
class PagedCase:
    q: torch.Tensor           # [B, H, dk]
    k_new: torch.Tensor       # [B, Hkv, dk]
    v_new: torch.Tensor       # [B, Hkv, dv]
    k_pool: torch.Tensor      # [num_blocks, Hkv, bs, dk]
    v_pool: torch.Tensor      # [num_blocks, Hkv, bs, dv]
    tables: torch.Tensor      # int32 [B, mbps], -1 past the used entries
    seq_lens: torch.Tensor    # int32 [B], history rows before the append
    scale: float
    theta: float
    block_size: int
    extras: dict = field(default_factory=dict)


def make_prefill(B=1, S=2048, H=14, Hkv=2, dk=64, dv=64, dtype=torch.bfloat16, seed=1,
                 device="cpu", offsets=None, S_kv=None, scale=None, theta=1e6) -> PrefillCase:
    g = generator(seed, device)
    S_kv = S if S_kv is None else S_kv
    q = randn((B, S, H, dk), g, dtype, device)
    k = randn((B, Hkv, S_kv, dk), g, dtype, device)
    v = randn((B, Hkv, S_kv, dv), g, dtype, device)
    off = torch.zeros(B, dtype=torch.int32) if offsets is None else torch.as_tensor(offsets,
                                                                                    dtype=torch.int32)
    return PrefillCase(q, k, v, off.to(device), 1.0 / math.sqrt(dk) if scale is None else scale, theta)


def make_contig(B=64, H=32, Hkv=8, dk=128, dv=128, max_len=8192, len_lo=512, len_hi=8192,
                dtype=torch.bfloat16, seed=2, device="cpu", d_rot=0, scale=None, lens=None) -> ContigCase:
    g = generator(seed, device)
    gl = generator(seed + 1000)
    if lens is None:
        lens = torch.randint(len_lo, len_hi + 1, (B,), generator=gl, dtype=torch.int32)
    lens = torch.as_tensor(lens, dtype=torch.int32)
    q = randn((B, H, dk), g, dtype, device)
    k = randn((B, Hkv, max_len, dk - d_rot), g, dtype, device)
    v = randn((B, Hkv, max_len, dv), g, dtype, device)
    k_rot = randn((B, max_len, d_rot), g, dtype, device) if d_rot else None
    return ContigCase(q, k, v, lens.to(device), 1.0 / math.sqrt(dk) if scale is None else scale, k_rot)


def make_mla(B=32, H=128, d_nope=128, d_rot=64, dv=128, cache_len=4096, dtype=torch.bfloat16, seed=4,
             device="cpu") -> ContigCase:
    """MLA-shaped decode: group size 1, K row = [k_nope (per head) | k_rot (shared)]."""
    c = make_contig(B=B, H=H, Hkv=H, dk=d_nope + d_rot, dv=dv, max_len=cache_len,
                    lens=[cache_len] * B, dtype=dtype, seed=seed, device=device, d_rot=d_rot)
    return c


def make_paged(B=256, H=32, Hkv=8, dk=128, dv=128, block_size=16, num_blocks=600_000,
               len_lo=1, len_hi=32768, dtype=torch.bfloat16, seed=3, device="cpu", lens=None,
               theta=1e6, scale=None, mbps=None) -> PagedCase:
    """History lengths are drawn first; each sequence takes the next
    ceil((len+1)/bs) entries of a seeded permutation of the pool (room for the
    appended row), so tables are disjoint; the rest of each row is -1."""
    gl = generator(seed + 1000)
    if lens is None:
        lens = torch.randint(len_lo, len_hi + 1, (B,), generator=gl, dtype=torch.int32)
    lens = torch.as_tensor(lens, dtype=torch.int32)
    need = [(int(n) + 1 + block_size - 1) // block_size for n in lens]
    if mbps is None:
        mbps = (len_hi + 1 + block_size - 1) // block_size
    if sum(need) > num_blocks or max(need) > mbps:
        raise ValueError("pool too small for the drawn lengths")
    perm = torch.randperm(num_blocks, generator=gl).to(torch.int32)
    tables = torch.full((B, mbps), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        tables[b, :n] = perm[at:at + n]
        at += n
    g = generator(seed, device)
    k_pool = randn((num_blocks, Hkv, block_size, dk), g, dtype, device)
    v_pool = randn((num_blocks, Hkv, block_size, dv), g, dtype, device)
    q = randn((B, H, dk), g, dtype, device)
    k_new = randn((B, Hkv, dk), g, dtype, device)
    v_new = randn((B, Hkv, dv), g, dtype, device)
    return PagedCase(q, k_new, v_new, k_pool, v_pool, tables.to(device), lens.to(device),
                     1.0 / math.sqrt(dk) if scale is None else scale, theta, block_size)


@dataclass
class MlaAbsorbedCase:
    q: torch.Tensor           # [B, H, d_nope + d_rope], the unabsorbed query
    k_b: torch.Tensor         # [H, d_c, d_nope], nope slice -> latent
    v_b: torch.Tensor         # [H, d_v, d_c], latent -> value width
    latent: torch.Tensor      # [B, max_len, d_c + d_rope]: rows (c_j, k_rot_j)
    lens: torch.Tensor        # int32 [B]
    scale: float              # 1 / sqrt(d_nope + d_rope), the unabsorbed head width's


def make_mla_absorbed(B=32, H=128, d_nope=128, d_rope=64, d_c=512, d_v=128, max_len=4096, lens=None,
                      dtype=torch.bfloat16, seed=9, device="cpu") -> MlaAbsorbedCase:
    """Absorbed MLA decode at the MLA-shaped config's model shape: latent rows
    N(0, 1); synthetic projections k_b ~ N(0, 1/d_nope) and v_b ~ N(0, 1/d_c), so
    that q_abs and the output keep unit scale; every sequence at max_len rows
    unless `lens` is given."""
    g = generator(seed, device)
    q = randn((B, H, d_nope + d_rope), g, dtype, device)
    k_b = (randn((H, d_c, d_nope), g, torch.float32, device) / math.sqrt(d_nope)).to(dtype)
    v_b = (randn((H, d_v, d_c), g, torch.float32, device) / math.sqrt(d_c)).to(dtype)
    latent = randn((B, max_len, d_c + d_rope), g, dtype, device)
    lens = torch.full((B,), max_len, dtype=torch.int32) if lens is None else torch.as_tensor(lens, dtype=torch.int32)
    return MlaAbsorbedCase(q, k_b, v_b, latent, lens.to(device), 1.0 / math.sqrt(d_nope + d_rope))


def make_tiny(seed=0, device="cpu"):
    """The tiny fp32 case: H=4, Hkv=2, d=16, scale 1/4; an 8-row prefill and a
    ninth row (q, k, v) for the decode step after it."""
    g = generator(seed, device)
    pre = PrefillCase(randn((1, 8, 4, 16), g, torch.float32, device),
                      randn((1, 2, 9, 16), g, torch.float32, device),
                      randn((1, 2, 9, 16), g, torch.float32, device),
                      torch.zeros(1, dtype=torch.int32, device=device), 0.25)
    q9 = randn((1, 4, 16), g, torch.float32, device)
    return pre, q9


# Full-size workload descriptions (used for names and algorithmic byte/flop counts).
WORKLOADS = {
    "prefill": "causal prefill bf16: B=1, H=14, Hkv=2, d=64, S=2048, RoPE theta 1e6",
    "contig": "contiguous decode bf16: 64 seqs, H=32, Hkv=8, d=128, len U[512,8192]",
    "paged": ("paged decode bf16: 256 seqs, H=32, Hkv=8, d=128, bs=16, 600k-block pool, "
              "history U[1,32768] + 1 appended row"),
    "mla": "MLA-shaped decode bf16: 32 seqs, 128 heads, d_k=128+64 shared rot, d_v=128, len 4096",
    "prefill_paged": ("chunked prefill bf16 on the paged pool: 4 seqs, H=14, Hkv=2, d=64, bs=16, a 2048-row "
                      "chunk at offsets 0/2048/4096/6144 (history already in the pool)"),
    "prefill_d128": "causal prefill bf16 at the decode configs' head shape: B=1, H=32, Hkv=8, d=128, S=2048",
    "mla_absorbed": ("absorbed (latent) MLA decode bf16: 32 seqs, 128 heads, latent rows 512 + 64 rot, "
                     "d_nope=128, d_v=128, len 4096"),
    "prefill_mla": "MLA-shaped causal prefill bf16: B=1, H=32, group 1, d_k=192 (128 + 64 rot), d_v=128, S=2048",
    "prefill_paged_d128": ("chunked prefill bf16 on the paged pool at the decode configs' head shape: 4 seqs, "
                           "H=32, Hkv=8, d=128, bs=16, a 2048-row chunk at offsets 0/2048/4096/6144"),
}


def make_prefill_paged(offsets=(0, 2048, 4096, 6144), S=2048, H=14, Hkv=2, d=64, bs=16, spare=64, seed=6,
                       device="cpu"):
    """Chunked-prefill case on a paged pool: sequence b holds offsets[b] + S rows
    (its history and the chunk itself, already appended), scattered over blocks
    of a seeded permutation of the pool; entries past a sequence's last block are
    -1. Returns (q [B, S, H, d], k_pool, v_pool, tables, offsets, scale)."""
    B = len(offsets)
    need = [(o + S + bs - 1) // bs for o in offsets]
    mbps = max(need)
    nb = sum(need) + spare
    gl = generator(seed + 1000)
    perm = torch.randperm(nb, generator=gl).to(torch.int32)
    tables = torch.full((B, mbps), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        tables[b, :n] = perm[at:at + n]
        at += n
    g = generator(seed, device)
    q = randn((B, S, H, d), g, torch.bfloat16, device)
    k_pool = randn((nb, Hkv, bs, d), g, torch.bfloat16, device)
    v_pool = randn((nb, Hkv, bs, d), g, torch.bfloat16, device)
    off = torch.tensor(list(offsets), dtype=torch.int32)
    return q, k_pool, v_pool, tables.to(device), off.to(device), 1.0 / math.sqrt(d)
