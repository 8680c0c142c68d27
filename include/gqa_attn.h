/*
 * gqa_attn.h -- C ABI of libgqa_attn.so: causal grouped-query attention of new
 * query rows against a KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (kopitiam-runtime 0.2.4 src/attention.rs, module doc,
 * `repeat_kv_heads`, `causal_mask`, `attention_forward`):
 *   query head h reads KV head h / (H / Hkv);
 *   query row i sits at absolute position position_offset + i and sees keys
 *   0 ..= position_offset + i, never later ones;
 *   out = softmax_j(attention_scale * q . k_j) weighted sum of v_j.
 * One rule covers a multi-row prefill (offset 0) and a single-row decode step
 * (offset = rows cached before the step).
 *
 * Conventions shared by every call:
 *  - Every tensor argument is a DEVICE pointer on the current CUDA device,
 *    owned by the caller. The library neither keeps nor frees any of them and
 *    allocates no device memory. `stream` is a cudaStream_t (NULL = the legacy
 *    default stream); every call is asynchronous on it.
 *  - Element type: `dt` gives the type of q, k, v, pools and out alike
 *    (GQA_F32 = float, GQA_BF16 = bfloat16). Arithmetic is fp32 whatever `dt`.
 *  - Layouts are dense row-major with the shapes given below; head and row
 *    widths d_k, d_v must be multiples of 8 and every tensor pointer 16-byte
 *    aligned.
 *  - Supported head widths (d_k, d_v) of the attention calls: (16,16), (32,32),
 *    (64,64), (128,128), (256,256), (192,128); others return
 *    GQA_ERR_UNSUPPORTED. The absorbed MLA calls (their own section below) take
 *    a 512-wide latent with a 64-wide rotated part, bf16 only.
 *  - Errors a host check can see (null pointer, H % Hkv != 0, bad size or
 *    alignment, small workspace) are returned before anything is launched.
 *  - Errors only the device can see (a block-table entry outside
 *    [0, num_blocks), a sequence length outside its valid range, a bounded
 *    wait that ran out) skip the affected work without any out-of-range access
 *    and set a sticky device error word; attn_get_device_error() reads and
 *    clears it. Outputs of the affected sequences are then unspecified.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1,    /* a host-checkable argument is wrong */
  GQA_ERR_UNSUPPORTED = 2,    /* valid, but a shape this library has no kernel for */
  GQA_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
  GQA_ERR_WORKSPACE = 4,      /* workspace missing or smaller than required */
  GQA_ERR_DEVICE_BOUNDS = 5,  /* device saw an index or length out of range */
  GQA_ERR_DEVICE_TIMEOUT = 6  /* a bounded device wait gave up */
} gqa_status;

typedef enum { GQA_F32 = 0, GQA_BF16 = 1 } gqa_dtype;

/*
 * Causal prefill: seq_q new rows per sequence attend to the cache that already
 * holds them (kopitiam-runtime src/attention.rs, `attention_forward` and
 * `causal_mask`; position_offset is an explicit argument, never re-derived from
 * the cache, as that page's `attention_forward` doc requires).
 *
 *   q    [B, seq_q, H, d_k]           (token-major; heads are a reshape of the hidden axis)
 *   k    [B, Hkv, seq_kv_max, d_k]    (head-major, kopitiam's per-layer [n_kv, seq, d])
 *   v    [B, Hkv, seq_kv_max, d_v]
 *   position_offset  int32 [B] on the device, or NULL for all zeros
 *   out  [B, seq_q, H, d_v]
 * Row i of sequence b sees keys 0..=position_offset[b] + i; it requires
 * position_offset[b] + seq_q <= seq_kv_max (checked on the device).
 * bf16 with (d_k, d_v) = (64, 64), (128, 128) or (192, 128) runs on the tcgen05
 * tensor-core kernel; every other shape and f32 run on the SIMT kernel. No
 * workspace.
 */
gqa_status attn_prefill_causal(const void* q, const void* k, const void* v, void* out, int B, int seq_q,
                               int seq_kv_max, const int32_t* position_offset, int H, int Hkv, int d_k,
                               int d_v, float attention_scale, gqa_dtype dt, void* stream);

/*
 * Single-row decode against contiguous per-sequence caches (frink-models
 * src/decoder/attn_block.rs, `push_and_attend_row`, contiguous arms: the row
 * is pushed first, then the sequence attends over all it holds).
 *
 *   q        [B, H, d_k]
 *   k_cache  [B, Hkv, max_len, d_k - d_rot]
 *   v_cache  [B, Hkv, max_len, d_v]
 *   k_rot_shared  NULL (d_rot = 0), or [B, max_len, d_rot]: one rotated vector per
 *            position shared by every KV head, so that key row j of head h is
 *            concat(k_cache[b, h, j, :], k_rot_shared[b, j, :]) -- the MLA shape of
 *            frink-models src/mla/mod.rs (`naive_attention`, module doc point 2).
 *            Supported for (d_k, d_v, d_rot) = (192, 128, 64).
 *   seq_lens int32 [B]: rows present, the query's own row included; the query
 *            sits at position seq_lens[b] - 1. Valid range 1..max_len.
 *   out      [B, H, d_v]
 * workspace: device scratch of at least attn_decode_workspace_bytes(B, H, d_v,
 * max_len) bytes (may be NULL when that is 0); its contents need no
 * initialisation and are clobbered.
 */
gqa_status attn_decode_contig(const void* q, const void* k_cache, const void* v_cache,
                              const void* k_rot_shared, int d_rot, const int32_t* seq_lens, void* out,
                              int B, int max_len, int H, int Hkv, int d_k, int d_v,
                              float attention_scale, gqa_dtype dt, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Single-row decode against a paged pool shared by all sequences (frink-models
 * src/decoder/attn_block.rs, `push_and_attend_row`, paged arm: paging changes
 * where rows live and nothing else, so the result is bit-identical to
 * attn_decode_contig on the same history).
 *
 *   k_pool        [num_blocks, Hkv, block_size, d_k]
 *   v_pool        [num_blocks, Hkv, block_size, d_v]
 *   block_tables  int32 [B, max_blocks_per_seq]: row j of sequence b lives in
 *                 block block_tables[b][j / block_size], slot j % block_size.
 *                 Entries past the sequence's last block are never read.
 *   seq_lens      int32 [B], as for attn_decode_contig; valid range
 *                 1..max_blocks_per_seq * block_size.
 *   q [B, H, d_k], out [B, H, d_v]; workspace as for attn_decode_contig with
 *   max_len = max_blocks_per_seq * block_size.
 */
gqa_status attn_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                             const int32_t* block_tables, const int32_t* seq_lens, void* out, int B,
                             int max_blocks_per_seq, int num_blocks, int block_size, int H, int Hkv,
                             int d_k, int d_v, float attention_scale, gqa_dtype dt, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * The arms of the attention row (frink-models src/decoder/attn_block.rs,
 * `push_and_attend_row`: one kernel serves plain, windowed, softcapped and
 * sink-bearing layers and takes ALiBi slopes too; the pages print no formula,
 * so these are the readings implemented). With s_j = attention_scale * q.k_j for
 * a row at position p:
 *   softcap > 0        s_j <- softcap * tanh(s_j / softcap)
 *   alibi_slopes[h]    s_j <- s_j + alibi_slopes[h] * (j - p)
 *   window > 0         only keys p - window < j <= p are visible (causal keys
 *                      j <= p as always); rows below the window are never read
 *                      and their block-table entries never looked at
 *   sinks[h]           one more term exp(sinks[h] - m) in the softmax
 *                      denominator, none in the numerator
 * in that order, then the softmax. The pages' own model code leaves softcap
 * off when a layer has sinks; the library takes any combination.
 * `gqa_arms` is read on the host during the call; sinks and alibi_slopes are
 * device pointers to H floats (4-byte aligned) or NULL. A NULL `arms` pointer,
 * or window <= 0, softcap <= 0 and NULL arrays, is plain attention.
 * GQA_ERR_INVALID_ARG: softcap not finite, a misaligned array.
 */
typedef struct gqa_arms {
  int window;
  float softcap;
  const float* sinks;
  const float* alibi_slopes;
} gqa_arms;

/* attn_decode_contig / attn_decode_paged / attn_prefill_causal with the arms;
 * every other argument as there. Prefill with an arm on runs on the tensor-core
 * kernel for the shapes it takes (bf16, (d_k, d_v) = (64, 64), (128, 128),
 * (192, 128)) and on the SIMT kernel otherwise, like the plain call. */
gqa_status attn_decode_contig_ex(const void* q, const void* k_cache, const void* v_cache,
                                 const void* k_rot_shared, int d_rot, const int32_t* seq_lens, void* out,
                                 int B, int max_len, int H, int Hkv, int d_k, int d_v, float attention_scale,
                                 gqa_dtype dt, void* workspace, size_t workspace_bytes, const gqa_arms* arms,
                                 void* stream);
gqa_status attn_decode_paged_ex(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                                const int32_t* seq_lens, void* out, int B, int max_blocks_per_seq, int num_blocks,
                                int block_size, int H, int Hkv, int d_k, int d_v, float attention_scale,
                                gqa_dtype dt, void* workspace, size_t workspace_bytes, const gqa_arms* arms,
                                void* stream);
gqa_status attn_prefill_causal_ex(const void* q, const void* k, const void* v, void* out, int B, int seq_q,
                                  int seq_kv_max, const int32_t* position_offset, int H, int Hkv, int d_k, int d_v,
                                  float attention_scale, gqa_dtype dt, const gqa_arms* arms, void* stream);

/*
 * Chunked prefill against the paged pool: seq_q new rows of each sequence,
 * already appended to the pool, attend to everything the sequence holds up to
 * their own positions -- the causal rule of attn_prefill_causal (kopitiam-runtime
 * src/attention.rs, `attention_forward`, `causal_mask`: row i at position
 * position_offset + i sees keys 0 ..= position_offset + i) with the paged
 * addressing of attn_decode_paged (frink-models src/decoder/attn_block.rs,
 * `push_and_attend_row`, paged arm: paging changes where rows live and nothing
 * else, so the result is bit-identical to attn_prefill_causal on the same
 * history). A decode step is the case seq_q = 1.
 *
 *   q             [B, seq_q, H, d_k]; out [B, seq_q, H, d_v]
 *   k_pool        [num_blocks, Hkv, block_size, d_k]
 *   v_pool        [num_blocks, Hkv, block_size, d_v]
 *   block_tables  int32 [B, max_blocks_per_seq], as for attn_decode_paged;
 *                 entries of blocks that hold no key the rows see are never read
 *   position_offset  int32 [B] on the device, or NULL for all zeros; requires
 *                 position_offset[b] + seq_q <= max_blocks_per_seq * block_size
 *                 (checked on the device)
 * bf16 with (d_k, d_v) = (64, 64), (128, 128) or (192, 128), block_size a
 * multiple of 8 dividing 128, max_blocks_per_seq <= 4096 and no arm runs on the
 * tcgen05 tensor-core kernel
 * (each 128-key tile gathered block by block with TMA); every other case on the
 * SIMT kernel. No workspace.
 * GQA_ERR_INVALID_ARG also for seq_q > max_blocks_per_seq * block_size.
 */
gqa_status attn_prefill_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                              const int32_t* position_offset, void* out, int B, int seq_q, int max_blocks_per_seq,
                              int num_blocks, int block_size, int H, int Hkv, int d_k, int d_v, float attention_scale,
                              gqa_dtype dt, void* stream);
/* attn_prefill_paged with the arms (`gqa_arms`); kernel choice as attn_prefill_causal_ex. */
gqa_status attn_prefill_paged_ex(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                                 const int32_t* position_offset, void* out, int B, int seq_q, int max_blocks_per_seq,
                                 int num_blocks, int block_size, int H, int Hkv, int d_k, int d_v,
                                 float attention_scale, gqa_dtype dt, const gqa_arms* arms, void* stream);

/* Size of the fixed device scratch behind attn_decode_paged_static_workspace. */
#define GQA_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)

/*
 * attn_decode_paged without a caller-supplied workspace, for callers that cannot
 * allocate device memory: a program whose GPU memory is all handed out up front
 * by another component (a serving engine that reserves the free HBM for its KV
 * pool, say), a plugin in a framework that exposes no allocator, or a loop that
 * must not risk the implicit synchronisation cudaMalloc/cudaFree can bring. The
 * pages have no counterpart of this call; it exists for such callers only.
 *
 * Arguments, layouts, results and errors are those of attn_decode_paged. The
 * split-K scratch is a fixed GQA_STATIC_WORKSPACE_BYTES array in the library's
 * device data, held by every GPU that loads the library until the process
 * exits; the call allocates nothing and calls no allocating routine. A problem
 * that needs more scratch than that (attn_decode_workspace_bytes(B, H, d_v,
 * max_blocks_per_seq * block_size) > GQA_STATIC_WORKSPACE_BYTES) is rejected
 * with GQA_ERR_WORKSPACE before anything is launched.
 *
 * Set-up: the first call on a device (a call with B = 0 is enough, and does
 * nothing else) looks up the array's device address with that device current.
 * Under CUDA's lazy module loading, the default, that is also when the CUDA
 * runtime places the array in the device's memory, so make this first call
 * before the rest of the device's memory is reserved, and before any stream
 * capture begins. Later calls only read the cached address; first calls from
 * several host threads at once are safe.
 *
 * Every call shares the one array per device: two calls whose kernels overlap
 * on the GPU (different streams, no ordering between them) race on it and may
 * return wrong results. Calls ordered on one stream are safe; no contents need
 * clearing between them (each call resets what it reads before reading it).
 */
gqa_status attn_decode_paged_static_workspace(const void* q, const void* k_pool, const void* v_pool,
                                              const int32_t* block_tables, const int32_t* seq_lens, void* out,
                                              int B, int max_blocks_per_seq, int num_blocks, int block_size,
                                              int H, int Hkv, int d_k, int d_v, float attention_scale,
                                              gqa_dtype dt, void* stream);

/*
 * Paged append of one new row per sequence, with interleaved RoPE on q and k
 * (frink-models src/decoder/attn_block.rs, `attn_block_tail` then
 * `push_and_attend_row`: per-head RoPE at the row's position, the position read
 * before the push, then the push).
 *
 *   q      [B, H, d_k]     rotated in place at p = seq_lens_in[b]
 *   k_new  [B, Hkv, d_k]   rotated at p, then written to k_pool
 *   v_new  [B, Hkv, d_v]   written to v_pool unrotated
 *   written slot: block block_tables[b][p / block_size], row p % block_size
 *   seq_lens_out[b] = p + 1 (seq_lens_out may alias seq_lens_in)
 * RoPE: rope_theta <= 0 disables it; otherwise the rotated slice is
 * [rot_offset, rot_offset + rot_dim) of every head, pairs (2t, 2t+1) turned by
 * p * rope_theta^(-2t / rot_dim) (the angle is formed and reduced in fp64).
 * A sequence whose position or block entry is out of range is skipped (its
 * seq_lens_out[b] = seq_lens_in[b]) and the device error word is set.
 */
gqa_status kv_append_paged(void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                           const int32_t* block_tables, const int32_t* seq_lens_in,
                           int32_t* seq_lens_out, int B, int max_blocks_per_seq, int num_blocks,
                           int block_size, int H, int Hkv, int d_k, int d_v, double rope_theta,
                           int rot_offset, int rot_dim, gqa_dtype dt, void* stream);

/*
 * Interleaved RoPE in place (frink-models src/mla/mod.rs, module doc point 2 and
 * `rotate_pe`: adjacent pairs, ggml NORM layout; frink-models
 * src/decoder/attn_block.rs, per-head RoPE in `attn_block_tail`).
 *
 *   x          heads_outer == 0: [B, T, heads, d]; heads_outer == 1: [B, heads, T, d]
 *   positions  int32 [B, T]: the absolute position of token t of sequence b
 * The slice [rot_offset, rot_offset + rot_dim) of every head is rotated pairwise
 * by pos * theta^(-2t / rot_dim), t < rot_dim / 2. rot_dim must be even, theta > 0.
 */
gqa_status attn_rope_interleaved(void* x, const int32_t* positions, int B, int T, int heads, int d,
                                 int heads_outer, int rot_offset, int rot_dim, double theta,
                                 gqa_dtype dt, void* stream);

/*
 * attn_rope_interleaved on the queries and the keys of the same tokens in one
 * launch (the prefill's "RoPE on q and k first"): each pair's angle is formed
 * once and turns every head of both. The results are bit-identical to two
 * attn_rope_interleaved calls with the same arguments.
 *   q  q_heads_outer == 0: [B, T, heads_q, d]; 1: [B, heads_q, T, d]  (16-byte aligned)
 *   k  k_heads_outer == 0: [B, T, heads_k, d]; 1: [B, heads_k, T, d]  (16-byte aligned)
 * Same positions, slice, theta and dtype for both; q and k must not overlap.
 */
gqa_status attn_rope_interleaved_qk(void* q, void* k, const int32_t* positions, int B, int T, int heads_q,
                                    int heads_k, int d, int q_heads_outer, int k_heads_outer, int rot_offset,
                                    int rot_dim, double theta, gqa_dtype dt, void* stream);

/* Bytes of workspace attn_decode_contig / attn_decode_paged need for B
 * sequences of at most max_len_upper_bound rows (0 when no sequence that long
 * is split). With S = ceil(max_len_upper_bound / 2048) splits and U = B*H*S:
 * a 256-byte scheduling header, the split list (8*U bytes rounded up to 256),
 * then the partial results (U * (d_v + 2) floats). Host only; launches nothing. */
size_t attn_decode_workspace_bytes(int B, int H, int d_v, int max_len_upper_bound);

/* ---- MLA, absorbed (latent) form -------------------------------------------
 * frink-models src/mla/mod.rs, `absorbed_attention` and `MlaKvB::Split`: the
 * cache holds one latent row per position, (c_j, k_rot_j) of width d_c + d_r
 * (kv_lora_rank + qk_rope); each query head's nope slice is absorbed into the
 * latent space through k_b[h], every head attends to the same rows (MQA, group
 * H) with the row as key and c_j as value, and each head's weighted latent is
 * mapped to the value width through v_b[h]. The three steps are three calls:
 * mla_absorb_q, attn_decode_mla_absorbed, mla_unabsorb_out. All pointers are
 * device pointers owned by the caller; bf16 only (GQA_ERR_UNSUPPORTED for f32).
 */

/* q_abs[b, h, :d_c] = k_b[h] q[b, h, :d_nope] (fp32 accumulation, rounded to
 * bf16) and q_abs[b, h, d_c:] = q[b, h, d_nope:] (copied).
 *   q      [B, H, d_nope + d_rope]
 *   k_b    [H, d_c, d_nope]   (maps qk_nope to the latent space)
 *   q_abs  [B, H, d_c + d_rope], must not alias q.
 * d_nope and d_rope multiples of 8; q and k_b 16-byte aligned. */
gqa_status mla_absorb_q(const void* q, const void* k_b, void* q_abs, int B, int H, int d_nope, int d_rope,
                        int d_c, gqa_dtype dt, void* stream);

/* Decode attention over the latent cache:
 *   out_lat[b, h] = sum_j w_j c_j / sum_j w_j,  w_j = exp(attention_scale * q_abs[b, h] . latent[b, j]),
 * over the rows j < seq_lens[b] (the query's own row included, as for
 * attn_decode_contig), c_j = latent[b, j, :d_c].
 *   q_abs    [B, H, d_c + d_r]  (16-byte aligned)
 *   latent   [B, max_len, d_c + d_r]  (16-byte aligned; rows at or past seq_lens[b] may hold anything)
 *   seq_lens int32 [B], 1 <= seq_lens[b] <= max_len; a length outside that range
 *            gives a zero output row and sets the device error word (GQA_ERR_DEVICE_BOUNDS)
 *   out_lat  [B, H, d_c]  (16-byte aligned)
 * Tensor-core path for (d_c, d_r) = (512, 64), any H (tiles of 128 heads);
 * other widths return GQA_ERR_UNSUPPORTED. attention_scale > 0 (the unabsorbed
 * head width's, 1 / sqrt(qk_nope + qk_rope)). workspace: at least
 * attn_decode_mla_absorbed_workspace_bytes(B, H, d_c, max_len) bytes, 16-byte
 * aligned (NULL allowed when that is 0). */
gqa_status attn_decode_mla_absorbed(const void* q_abs, const void* latent, const int32_t* seq_lens, void* out_lat,
                                    int B, int max_len, int H, int d_c, int d_r, float attention_scale,
                                    gqa_dtype dt, void* workspace, size_t workspace_bytes, void* stream);

/* attn_decode_mla_absorbed over a paged latent cache: row j of sequence b is
 * latent_pool[block_tables[b * max_blocks_per_seq + j / block_size], j % block_size]
 * (the paged addressing of attn_decode_paged with one latent row per slot).
 *   latent_pool  [num_blocks, block_size, d_c + d_r]  (16-byte aligned)
 *   block_tables int32 [B, max_blocks_per_seq]; entries past a sequence's rows are never read
 *   seq_lens     1 <= seq_lens[b] <= max_blocks_per_seq * block_size
 * block_size one of 8, 16, 32, 64 (else GQA_ERR_UNSUPPORTED). A table entry outside
 * [0, num_blocks) for a visible row sets GQA_ERR_DEVICE_BOUNDS and its rows read as
 * zeros. Same arithmetic as the contiguous call: the outputs are bit-identical to
 * it on the same rows when max_blocks_per_seq * block_size equals its max_len
 * (the capacity decides the split size). Workspace: attn_decode_mla_absorbed_workspace_bytes(B, H, d_c,
 * max_blocks_per_seq * block_size). */
gqa_status attn_decode_mla_absorbed_paged(const void* q_abs, const void* latent_pool, const int32_t* block_tables,
                                          const int32_t* seq_lens, void* out_lat, int B, int max_blocks_per_seq,
                                          int num_blocks, int block_size, int H, int d_c, int d_r,
                                          float attention_scale, gqa_dtype dt, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* Workspace of attn_decode_mla_absorbed: rows are split C at a time, C = 1024
 * doubled (up to 8192) while B * ceil(H / 128) * ceil(max_len / (2 C)) >= 64;
 * with S = ceil(max_len / C) > 1 splits, B * H * S * (d_c + 2) floats, else 0.
 * C depends on B, H and max_len only (max_blocks_per_seq * block_size for the
 * paged call). Host only. */
size_t attn_decode_mla_absorbed_workspace_bytes(int B, int H, int d_c, int max_len);

/* out[b, h] = v_b[h] out_lat[b, h] (fp32 accumulation, rounded to bf16).
 *   out_lat [B, H, d_c], v_b [H, d_v, d_c], out [B, H, d_v], must not alias out_lat.
 * d_c a multiple of 8; out_lat and v_b 16-byte aligned. */
gqa_status mla_unabsorb_out(const void* out_lat, const void* v_b, void* out, int B, int H, int d_c, int d_v,
                            gqa_dtype dt, void* stream);

/* Synchronises `stream`, then returns and clears the device error word of the
 * current device: GQA_OK, GQA_ERR_DEVICE_TIMEOUT (takes precedence) or
 * GQA_ERR_DEVICE_BOUNDS; GQA_ERR_CUDA if the stream reports a CUDA error. */
gqa_status attn_get_device_error(void* stream);

/* Static, NUL-terminated text of a status code. */
const char* gqa_status_string(gqa_status status);

/* Test hook for the bounded waits: while enabled, the kernels with a TMA
 * producer never request one of their copies, so that the wait on it runs out
 * (after about one second), the device error word records
 * GQA_ERR_DEVICE_TIMEOUT and the kernel returns with nothing in flight and its
 * tensor memory released:
 *   - the SIMT attention kernel (decode; SIMT prefill): the first K/V tile of
 *     every CTA;
 *   - the tensor-core prefill: the first K tile of every CTA;
 *   - the absorbed MLA decode: the first cache tile of the second CTA of every
 *     pair, so the first CTA also gives up waiting for its peer's tile maxima;
 *     both let what they sent each other land before releasing their memory.
 * Outputs are then garbage. The hook is read when a call launches.
 * Never enable outside tests. Returns the previous setting. */
int gqa_debug_withhold_first_tile(int enable);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
