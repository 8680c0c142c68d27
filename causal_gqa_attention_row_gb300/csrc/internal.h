// internal.h -- host-side declarations shared by the translation units of
// libgqa_attn.so (not part of the public ABI; see include/gqa_attn.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gqa {

// Bits of the device error word.
enum : unsigned { kErrBounds = 1u, kErrTimeout = 2u };

// Rows of one split-K work item. Split boundaries are multiples of this, a
// fixed number independent of the layout and of the rest of the batch, so the
// paged and contiguous decodes of one history do identical arithmetic.
constexpr int kSplitRows = 2048;

// Parameters of the SIMT attention kernel (decode, and prefill shapes that the
// tensor-core kernel does not take). All pointers are device pointers.
struct RowsParams {
  const void* q;            // [B, seq_q, H, DK]
  const void* k;            // contiguous [B, Hkv, max_len, DK-DROT] or pool [nb, Hkv, bs, DK]
  const void* v;            // contiguous [B, Hkv, max_len, DV] or pool [nb, Hkv, bs, DV]
  const void* k_rot;        // contiguous only: [B, max_len, DROT]
  void* out;                // [B, seq_q, H, DV]
  float* partial;           // [B*seq_q*H, max_splits, DV+2] when max_splits > 1
  int* sched;               // split-K plan: [0] ticket counter, [1] units listed; NULL without a workspace
  int2* units;              // split-K plan: the listed (item, split) units
  const int32_t* kv_len;    // [B] keys present (decode), or NULL: offsets[b] + seq_q
  const int32_t* offsets;   // [B] or NULL (prefill)
  const int32_t* tables;    // paged: [B, mbps]
  unsigned* err;            // device error word
  int paged;
  int B, seq_q, H, Hkv, G;  // G = H / Hkv
  int GH, QR;               // query heads and query rows per work item (GH*QR = NV)
  int n_hchunks, n_rblocks; // G / GH, ceil(seq_q / QR)
  int max_len;              // contiguous rows per (b, kvh); 0 when paged
  int capacity;             // largest valid key count of one sequence
  int mbps, bs, num_blocks; // paged
  int split_rows;           // rows per split (kSplitRows, or >= capacity for no split)
  int max_splits;
  float qscale;             // attention_scale * log2(e)
  int debug_withhold;       // test hook: withhold the first tile of every CTA
  // The arms of the attention row (all off when zero / NULL): a row at
  // position p sees keys first_visible_key(p, window)..p; scores s (natural
  // units) become softcap * tanh(s / softcap), then s + alibi[h] * (j - p); the
  // sink logit sinks[h] joins the softmax denominator only.
  int window;               // > 0: the last `window` positions; <= 0: no window
  float softcap2;           // softcap * log2(e) (the kernels score in the log2 domain); 0: none
  const float* sinks;       // [H] device, natural units, or NULL
  const float* alibi;       // [H] device, natural units, or NULL
};

constexpr float kLog2e = 1.4426950408889634f;

// First key a row at position p sees: p - window + 1 (not below 0) with a
// window, else 0.
__host__ __device__ inline int first_visible_key(int p, int window) {
  return (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
}

// Dispatch of the SIMT kernel by element type and head widths; NV = GH * QR.
// Returns cudaErrorNotSupported when there is no instantiation.
cudaError_t launch_attn_rows_f32(const RowsParams& p, int dk, int dv, int drot, int nv, cudaStream_t st);
cudaError_t launch_attn_rows_bf16(const RowsParams& p, int dk, int dv, int drot, int nv, cudaStream_t st);
// Largest NV the instantiation set offers for these widths (0 = unsupported).
int rows_max_nv(int bf16, int dk, int dv, int drot);

cudaError_t launch_split_combine(const RowsParams& p, int dv, int bf16, cudaStream_t st);

// The split-K plan: lists the units with keys into p.units and resets the
// ticket counter (p.sched must be set).
cudaError_t launch_plan_units(const RowsParams& p, cudaStream_t st);

// Split-K workspace layout: the plan (ticket counter and total, then the unit
// list), then the partial results.
constexpr size_t kPlanHeaderBytes = 256;
inline size_t round_up256(size_t n) { return (n + 255) / 256 * 256; }
inline size_t plan_bytes(size_t units_max) { return kPlanHeaderBytes + round_up256(units_max * 8); }

// x2 != NULL: a second tensor of the same tokens (heads2 heads, its own layout)
// turned by the same angles in the same launch.
cudaError_t launch_rope(void* x, const int32_t* positions, int B, int T, int heads, int d, int heads_outer,
                        int rot_offset, int rot_dim, double theta, int bf16, cudaStream_t st, void* x2 = nullptr,
                        int heads2 = 0, int heads_outer2 = 0);

cudaError_t launch_append(void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                          const int32_t* tables, const int32_t* lens_in, int32_t* lens_out, int B, int mbps,
                          int num_blocks, int bs, int H, int Hkv, int dk, int dv, double theta, int rot_offset,
                          int rot_dim, int bf16, unsigned* err, cudaStream_t st);

// The arms for the tensor-core prefill: window (<= 0: none), softcap * log2 e
// (0: none), sink logits and ALiBi slopes ([H] fp32 on the device, natural
// units, or NULL).
struct TcArms {
  int window;
  float softcap2;
  const float* sinks;
  const float* alibi;
};

// tcgen05 causal prefill (bf16, d_k = d_v = 64). Returns cudaErrorNotSupported
// for other shapes. Contiguous k, v [B, Hkv, seq_kv_max, 64] (tables NULL), or
// paged pools [num_blocks, Hkv, bs, 64] with block tables [B, mbps] and
// seq_kv_max = mbps * bs.
cudaError_t launch_prefill_tc(const void* q, const void* k, const void* v, void* out, int B, int seq_q,
                              int seq_kv_max, const int32_t* offsets, int H, int Hkv, int dk, int dv,
                              float qscale, unsigned* err, cudaStream_t st, const int32_t* tables = nullptr,
                              int mbps = 0, int bs = 0, int num_blocks = 0, const TcArms* arms = nullptr,
                              int debug_withhold = 0);
// bs = 0: contiguous K/V; else the pool's block size and max blocks per sequence.
bool prefill_tc_supported(int bf16, int dk, int dv, int bs = 0, int mbps = 0);

// Absorbed MLA decode on tcgen05 (bf16, d_c = 512, d_r = 64): attention of
// q_abs [B, H, d_c + d_r] over the latent rows [B, max_len, d_c + d_r] (value =
// the first d_c columns) into out_lat [B, H, d_c]; splits of `chunk` rows write
// (m, l, o) into partial [B * H, ceil(max_len / chunk), d_c + 2] when a sequence
// has more than one, and the split combine merges them.
bool mla_absorbed_tc_supported(int bf16, int d_c, int d_r);
// Paged (tables != NULL): latent is a pool [num_blocks, bs, d_c + d_r], max_len
// is ignored (mbps * bs rows per sequence), bs one of 8, 16, 32, 64.
cudaError_t launch_mla_absorbed_tc(const void* q_abs, const void* latent, const int32_t* seq_lens, void* out_lat,
                                   float* partial, int B, int max_len, int H, int d_c, int d_r, int chunk,
                                   float qscale, unsigned* err, cudaStream_t st, const int32_t* tables = nullptr,
                                   int mbps = 0, int bs = 0, int num_blocks = 0, int debug_withhold = 0);
bool mla_absorbed_paged_block_ok(int bs);
// Rows of one split of the absorbed MLA decode: 1024, doubled (up to 8192) while
// the (sequence, head tile, split) clusters of a call at its capacity would still
// number at least 64 (one wave of the GPU's 76 two-CTA cluster slots, nearly
// filled), so that a batch fills the GPU with as few partial results to merge
// as it can. A function of B, H and the capacity alone: a sequence's result does
// not depend on the lengths of the others, and two calls with the same three
// values split alike.
constexpr int kMlaChunk = 1024;
inline int mla_chunk_rows(int B, int H, int capacity) {
  const long long clusters_per_split = (long long)B * ((H + 127) / 128);
  int chunk = kMlaChunk;
  while (chunk < 8192 && clusters_per_split * (((long long)capacity + 2 * chunk - 1) / (2 * chunk)) >= 64) chunk *= 2;
  return chunk;
}

// y[b, h, :M] = W[h] x[b, h, :K] (bf16, fp32 accumulation), W [H, M, K]; the
// `tail` columns of x after K are copied to y after M.
cudaError_t launch_head_matvec(const void* W, const void* x, int x_stride, void* y, int y_stride, int B, int H, int M,
                               int K, int tail, cudaStream_t st);

// The same product on tcgen05 (bf16): W's rows in tiles of 128 (M % 128 == 0),
// K % 64 == 0 and K <= 512; cudaErrorNotSupported otherwise.
bool head_proj_tc_supported(int M, int K);
cudaError_t launch_head_proj_tc(const void* W, const void* x, int x_stride, void* y, int y_stride, int B, int H, int M,
                                int K, int tail, unsigned* err, cudaStream_t st);

}  // namespace gqa
