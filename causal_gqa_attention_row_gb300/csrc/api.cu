// api.cu -- the extern "C" entry points of libgqa_attn.so (include/gqa_attn.h):
// host-side argument checks, work decomposition, and launches. No device
// memory is allocated here; the only device state is the error word below.
#include <atomic>
#include <cmath>
#include <climits>
#include <cstdint>

#include "gqa_attn.h"
#include "internal.h"

// Sticky device error word (bits gqa::kErrBounds, gqa::kErrTimeout), one per
// device that loads the library. Kernels in other translation units receive its
// device address as a parameter.
__device__ unsigned int g_gqa_error_word = 0;

namespace {

int g_withhold_first_tile = 0;

// Device address of the error word on the current device, looked up once per
// device; the cache is atomic, so concurrent first calls from several host
// threads are safe (each stores the same value).
unsigned* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static std::atomic<void*> cache[64];
  void* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_gqa_error_word) != cudaSuccess || p == nullptr) return nullptr;
    cache[dev].store(p, std::memory_order_release);
  }
  return static_cast<unsigned*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool heads_ok(int H, int Hkv) { return H > 0 && Hkv > 0 && H % Hkv == 0; }

bool width_ok(int d) { return d > 0 && d % 8 == 0 && d <= 256; }

int dtype_flag(gqa_dtype dt) { return dt == GQA_BF16 ? 1 : (dt == GQA_F32 ? 0 : -1); }

// Largest power of two <= cap that divides n.
int pow2_divisor(int n, int cap) {
  int g = 1;
  while (g * 2 <= cap && n % (g * 2) == 0) g *= 2;
  return g;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

gqa_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return GQA_OK;
  if (e == cudaErrorNotSupported) return GQA_ERR_UNSUPPORTED;
  return GQA_ERR_CUDA;
}

gqa_status launch_rows(const gqa::RowsParams& p, int bf16, int dk, int dv, int drot, int nv, cudaStream_t st) {
  if (p.sched) {
    const cudaError_t ep = gqa::launch_plan_units(p, st);
    if (ep != cudaSuccess) return from_cuda(ep);
  }
  cudaError_t e = bf16 ? gqa::launch_attn_rows_bf16(p, dk, dv, drot, nv, st)
                       : gqa::launch_attn_rows_f32(p, dk, dv, drot, nv, st);
  if (e != cudaSuccess) return from_cuda(e);
  if (p.max_splits > 1) return from_cuda(gqa::launch_split_combine(p, dv, bf16, st));
  return GQA_OK;
}

// The arms of the attention row into the kernel parameters; true when any is on.
gqa_status apply_arms(gqa::RowsParams& p, const gqa_arms* arms, bool* active) {
  *active = false;
  if (!arms) return GQA_OK;
  if (!std::isfinite(arms->softcap)) return GQA_ERR_INVALID_ARG;
  if ((arms->sinks && reinterpret_cast<uintptr_t>(arms->sinks) % 4) ||
      (arms->alibi_slopes && reinterpret_cast<uintptr_t>(arms->alibi_slopes) % 4))
    return GQA_ERR_INVALID_ARG;
  p.window = arms->window > 0 ? arms->window : 0;
  p.softcap2 = arms->softcap > 0.f ? arms->softcap * gqa::kLog2e : 0.f;
  p.sinks = arms->sinks;
  p.alibi = arms->alibi_slopes;
  *active = p.window > 0 || p.softcap2 > 0.f || p.sinks || p.alibi;
  return GQA_OK;
}

}  // namespace

extern "C" {

size_t attn_decode_workspace_bytes(int B, int H, int d_v, int max_len_upper_bound) {
  if (B <= 0 || H <= 0 || d_v <= 0 || max_len_upper_bound <= gqa::kSplitRows) return 0;
  const size_t splits = (size_t)ceil_div(max_len_upper_bound, gqa::kSplitRows);
  const size_t units = (size_t)B * (size_t)H * splits;  // at least the (item, split) units of a call
  return gqa::plan_bytes(units) + units * (size_t)(d_v + 2) * sizeof(float);
}

static gqa_status decode_common(gqa::RowsParams& p, int bf16, int d_k, int d_v, int d_rot, void* workspace,
                                size_t workspace_bytes, cudaStream_t st) {
  const int nvmax = gqa::rows_max_nv(bf16, d_k, d_v, d_rot);
  if (nvmax == 0) return GQA_ERR_UNSUPPORTED;
  p.G = p.H / p.Hkv;
  p.GH = pow2_divisor(p.G, nvmax);
  p.QR = 1;
  p.n_hchunks = p.G / p.GH;
  p.n_rblocks = 1;
  p.seq_q = 1;
  p.split_rows = gqa::kSplitRows;
  p.max_splits = ceil_div(p.capacity, gqa::kSplitRows);
  const size_t need = attn_decode_workspace_bytes(p.B, p.H, d_v, p.capacity);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return GQA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GQA_ERR_INVALID_ARG;
  }
  if (need > 0) {
    const size_t units = (size_t)p.B * (size_t)p.H * (size_t)p.max_splits;
    p.sched = static_cast<int*>(workspace);
    p.units = reinterpret_cast<int2*>(static_cast<char*>(workspace) + gqa::kPlanHeaderBytes);
    p.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + gqa::plan_bytes(units));
  }
  p.err = error_word();
  if (!p.err) return GQA_ERR_CUDA;
  p.debug_withhold = g_withhold_first_tile;
  return launch_rows(p, bf16, d_k, d_v, d_rot, p.GH, st);
}

gqa_status attn_decode_contig_ex(const void* q, const void* k_cache, const void* v_cache, const void* k_rot_shared,
                                 int d_rot, const int32_t* seq_lens, void* out, int B, int max_len, int H, int Hkv,
                                 int d_k, int d_v, float attention_scale, gqa_dtype dt, void* workspace,
                                 size_t workspace_bytes, const gqa_arms* arms, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || max_len <= 0 || !heads_ok(H, Hkv) || !width_ok(d_k) || !width_ok(d_v))
    return GQA_ERR_INVALID_ARG;
  if (d_rot < 0 || d_rot >= d_k || d_rot % 8 || (k_rot_shared == nullptr) != (d_rot == 0))
    return GQA_ERR_INVALID_ARG;
  if (B == 0) return GQA_OK;
  if (!q || !k_cache || !v_cache || !seq_lens || !out) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (k_rot_shared && !aligned16(k_rot_shared)))
    return GQA_ERR_INVALID_ARG;
  gqa::RowsParams p{};
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.k_rot = k_rot_shared;
  p.out = out;
  p.kv_len = seq_lens;
  p.paged = 0;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.max_len = max_len;
  p.capacity = max_len;
  p.qscale = attention_scale * 1.4426950408889634f;
  bool arms_on;
  const gqa_status sa = apply_arms(p, arms, &arms_on);
  if (sa != GQA_OK) return sa;
  return decode_common(p, bf16, d_k, d_v, d_rot, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

gqa_status attn_decode_paged_ex(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                                const int32_t* seq_lens, void* out, int B, int max_blocks_per_seq, int num_blocks,
                                int block_size, int H, int Hkv, int d_k, int d_v, float attention_scale,
                                gqa_dtype dt, void* workspace, size_t workspace_bytes, const gqa_arms* arms,
                                void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0 || !heads_ok(H, Hkv) ||
      !width_ok(d_k) || !width_ok(d_v))
    return GQA_ERR_INVALID_ARG;
  if ((long long)max_blocks_per_seq * block_size > INT_MAX / 2) return GQA_ERR_INVALID_ARG;
  if (B == 0) return GQA_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return GQA_ERR_INVALID_ARG;
  gqa::RowsParams p{};
  p.q = q;
  p.k = k_pool;
  p.v = v_pool;
  p.out = out;
  p.kv_len = seq_lens;
  p.tables = block_tables;
  p.paged = 1;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.max_len = 0;
  p.capacity = max_blocks_per_seq * block_size;
  p.mbps = max_blocks_per_seq;
  p.bs = block_size;
  p.num_blocks = num_blocks;
  p.qscale = attention_scale * 1.4426950408889634f;
  bool arms_on;
  const gqa_status sa = apply_arms(p, arms, &arms_on);
  if (sa != GQA_OK) return sa;
  return decode_common(p, bf16, d_k, d_v, 0, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

// Prefill, contiguous or paged (p holds the pointers, shapes and arms): the
// tcgen05 kernel for the shapes it takes, else the SIMT kernel with one split
// per work item (every item covers its whole key range; no workspace).
static gqa_status prefill_common(gqa::RowsParams& p, int bf16, int d_k, int d_v, float attention_scale, bool arms_on,
                                 cudaStream_t st) {
  p.err = error_word();
  if (!p.err) return GQA_ERR_CUDA;
  const float qscale = attention_scale * 1.4426950408889634f;
  if (gqa::prefill_tc_supported(bf16, d_k, d_v, p.paged ? p.bs : 0, p.mbps) && attention_scale > 0.f) {
    const gqa::TcArms tc_arms{p.window, p.softcap2, p.sinks, p.alibi};
    return from_cuda(gqa::launch_prefill_tc(p.q, p.k, p.v, p.out, p.B, p.seq_q, p.capacity, p.offsets, p.H, p.Hkv,
                                            d_k, d_v, qscale, p.err, st, p.paged ? p.tables : nullptr, p.mbps, p.bs,
                                            p.num_blocks, arms_on ? &tc_arms : nullptr, g_withhold_first_tile));
  }
  const int nvmax = gqa::rows_max_nv(bf16, d_k, d_v, 0);
  if (nvmax == 0) return GQA_ERR_UNSUPPORTED;
  p.G = p.H / p.Hkv;
  p.GH = pow2_divisor(p.G, nvmax);
  p.QR = 1;
  while (p.GH * p.QR * 2 <= nvmax && p.QR < p.seq_q) p.QR *= 2;
  p.n_hchunks = p.G / p.GH;
  p.n_rblocks = ceil_div(p.seq_q, p.QR);
  p.split_rows = p.capacity;
  p.max_splits = 1;
  p.qscale = qscale;
  return launch_rows(p, bf16, d_k, d_v, 0, p.GH * p.QR, st);
}

gqa_status attn_prefill_causal_ex(const void* q, const void* k, const void* v, void* out, int B, int seq_q,
                                  int seq_kv_max, const int32_t* position_offset, int H, int Hkv, int d_k, int d_v,
                                  float attention_scale, gqa_dtype dt, const gqa_arms* arms, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || seq_q < 0 || seq_kv_max <= 0 || seq_q > seq_kv_max || !heads_ok(H, Hkv) ||
      !width_ok(d_k) || !width_ok(d_v))
    return GQA_ERR_INVALID_ARG;
  if (B == 0 || seq_q == 0) return GQA_OK;
  if (!q || !k || !v || !out) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return GQA_ERR_INVALID_ARG;
  gqa::RowsParams p{};
  bool arms_on;
  const gqa_status sa = apply_arms(p, arms, &arms_on);
  if (sa != GQA_OK) return sa;
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.offsets = position_offset;
  p.paged = 0;
  p.B = B;
  p.seq_q = seq_q;
  p.H = H;
  p.Hkv = Hkv;
  p.max_len = seq_kv_max;
  p.capacity = seq_kv_max;
  return prefill_common(p, bf16, d_k, d_v, attention_scale, arms_on, static_cast<cudaStream_t>(stream));
}

gqa_status attn_prefill_paged_ex(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                                 const int32_t* position_offset, void* out, int B, int seq_q, int max_blocks_per_seq,
                                 int num_blocks, int block_size, int H, int Hkv, int d_k, int d_v,
                                 float attention_scale, gqa_dtype dt, const gqa_arms* arms, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || seq_q < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0 ||
      !heads_ok(H, Hkv) || !width_ok(d_k) || !width_ok(d_v))
    return GQA_ERR_INVALID_ARG;
  if ((long long)max_blocks_per_seq * block_size > INT_MAX / 2) return GQA_ERR_INVALID_ARG;
  if (seq_q > max_blocks_per_seq * block_size) return GQA_ERR_INVALID_ARG;
  if (B == 0 || seq_q == 0) return GQA_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !out) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return GQA_ERR_INVALID_ARG;
  gqa::RowsParams p{};
  bool arms_on;
  const gqa_status sa = apply_arms(p, arms, &arms_on);
  if (sa != GQA_OK) return sa;
  p.q = q;
  p.k = k_pool;
  p.v = v_pool;
  p.out = out;
  p.offsets = position_offset;
  p.tables = block_tables;
  p.paged = 1;
  p.B = B;
  p.seq_q = seq_q;
  p.H = H;
  p.Hkv = Hkv;
  p.max_len = 0;
  p.capacity = max_blocks_per_seq * block_size;
  p.mbps = max_blocks_per_seq;
  p.bs = block_size;
  p.num_blocks = num_blocks;
  return prefill_common(p, bf16, d_k, d_v, attention_scale, arms_on, static_cast<cudaStream_t>(stream));
}

// The plain calls: the _ex calls with no arms.
gqa_status attn_decode_contig(const void* q, const void* k_cache, const void* v_cache, const void* k_rot_shared,
                              int d_rot, const int32_t* seq_lens, void* out, int B, int max_len, int H, int Hkv,
                              int d_k, int d_v, float attention_scale, gqa_dtype dt, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return attn_decode_contig_ex(q, k_cache, v_cache, k_rot_shared, d_rot, seq_lens, out, B, max_len, H, Hkv, d_k, d_v,
                               attention_scale, dt, workspace, workspace_bytes, nullptr, stream);
}

gqa_status attn_decode_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                             const int32_t* seq_lens, void* out, int B, int max_blocks_per_seq, int num_blocks,
                             int block_size, int H, int Hkv, int d_k, int d_v, float attention_scale, gqa_dtype dt,
                             void* workspace, size_t workspace_bytes, void* stream) {
  return attn_decode_paged_ex(q, k_pool, v_pool, block_tables, seq_lens, out, B, max_blocks_per_seq, num_blocks,
                              block_size, H, Hkv, d_k, d_v, attention_scale, dt, workspace, workspace_bytes, nullptr,
                              stream);
}

gqa_status attn_prefill_causal(const void* q, const void* k, const void* v, void* out, int B, int seq_q,
                               int seq_kv_max, const int32_t* position_offset, int H, int Hkv, int d_k, int d_v,
                               float attention_scale, gqa_dtype dt, void* stream) {
  return attn_prefill_causal_ex(q, k, v, out, B, seq_q, seq_kv_max, position_offset, H, Hkv, d_k, d_v,
                                attention_scale, dt, nullptr, stream);
}

gqa_status attn_prefill_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                              const int32_t* position_offset, void* out, int B, int seq_q, int max_blocks_per_seq,
                              int num_blocks, int block_size, int H, int Hkv, int d_k, int d_v, float attention_scale,
                              gqa_dtype dt, void* stream) {
  return attn_prefill_paged_ex(q, k_pool, v_pool, block_tables, position_offset, out, B, seq_q, max_blocks_per_seq,
                               num_blocks, block_size, H, Hkv, d_k, d_v, attention_scale, dt, nullptr, stream);
}

gqa_status kv_append_paged(void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                           const int32_t* block_tables, const int32_t* seq_lens_in, int32_t* seq_lens_out, int B,
                           int max_blocks_per_seq, int num_blocks, int block_size, int H, int Hkv, int d_k, int d_v,
                           double rope_theta, int rot_offset, int rot_dim, gqa_dtype dt, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0 || !heads_ok(H, Hkv) ||
      d_k <= 0 || d_v <= 0 || d_k % 2)
    return GQA_ERR_INVALID_ARG;
  if (rope_theta > 0.0 && (rot_dim <= 0 || rot_dim % 2 || rot_offset < 0 || rot_offset + rot_dim > d_k))
    return GQA_ERR_INVALID_ARG;
  if ((long long)max_blocks_per_seq * block_size > INT_MAX / 2) return GQA_ERR_INVALID_ARG;
  if (B == 0) return GQA_OK;
  if (!q || !k_new || !v_new || !k_pool || !v_pool || !block_tables || !seq_lens_in || !seq_lens_out)
    return GQA_ERR_INVALID_ARG;
  unsigned* err = error_word();
  if (!err) return GQA_ERR_CUDA;
  return from_cuda(gqa::launch_append(q, k_new, v_new, k_pool, v_pool, block_tables, seq_lens_in, seq_lens_out, B,
                                      max_blocks_per_seq, num_blocks, block_size, H, Hkv, d_k, d_v, rope_theta,
                                      rot_offset, rope_theta > 0.0 ? rot_dim : 0, bf16, err,
                                      static_cast<cudaStream_t>(stream)));
}

gqa_status attn_rope_interleaved(void* x, const int32_t* positions, int B, int T, int heads, int d, int heads_outer,
                                 int rot_offset, int rot_dim, double theta, gqa_dtype dt, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || T < 0 || heads <= 0 || d <= 0 || d % 2 || rot_dim <= 0 || rot_dim % 2 ||
      rot_offset < 0 || rot_offset % 2 || rot_offset + rot_dim > d || !(theta > 0.0) ||
      (heads_outer != 0 && heads_outer != 1))
    return GQA_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return GQA_OK;
  if (!x || !positions || !aligned16(x)) return GQA_ERR_INVALID_ARG;
  return from_cuda(gqa::launch_rope(x, positions, B, T, heads, d, heads_outer, rot_offset, rot_dim, theta, bf16,
                                    static_cast<cudaStream_t>(stream)));
}

gqa_status attn_rope_interleaved_qk(void* q, void* k, const int32_t* positions, int B, int T, int heads_q, int heads_k,
                                    int d, int q_heads_outer, int k_heads_outer, int rot_offset, int rot_dim,
                                    double theta, gqa_dtype dt, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || T < 0 || heads_q <= 0 || heads_k <= 0 || d <= 0 || d % 2 || rot_dim <= 0 ||
      rot_dim % 2 || rot_offset < 0 || rot_offset % 2 || rot_offset + rot_dim > d || !(theta > 0.0) ||
      (q_heads_outer != 0 && q_heads_outer != 1) || (k_heads_outer != 0 && k_heads_outer != 1))
    return GQA_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return GQA_OK;
  if (!q || !k || !positions || !aligned16(q) || !aligned16(k)) return GQA_ERR_INVALID_ARG;
  return from_cuda(gqa::launch_rope(q, positions, B, T, heads_q, d, q_heads_outer, rot_offset, rot_dim, theta, bf16,
                                    static_cast<cudaStream_t>(stream), k, heads_k, k_heads_outer));
}

size_t attn_decode_mla_absorbed_workspace_bytes(int B, int H, int d_c, int max_len) {
  if (B <= 0 || H <= 0 || d_c <= 0 || max_len <= 0) return 0;
  const int chunk = gqa::mla_chunk_rows(B, H, max_len);
  if (max_len <= chunk) return 0;
  const size_t splits = (size_t)ceil_div(max_len, chunk);
  return (size_t)B * (size_t)H * splits * (size_t)(d_c + 2) * sizeof(float);
}

// The absorbed MLA decode, contiguous latent cache (tables NULL) or paged pool.
static gqa_status mla_absorbed_common(const void* q_abs, const void* latent, const int32_t* seq_lens, void* out_lat,
                                      int B, int capacity, int H, int d_c, int d_r, float attention_scale, int bf16,
                                      void* workspace, size_t workspace_bytes, cudaStream_t st,
                                      const int32_t* tables, int mbps, int bs, int num_blocks) {
  if (!gqa::mla_absorbed_tc_supported(bf16, d_c, d_r) || !(attention_scale > 0.f)) return GQA_ERR_UNSUPPORTED;
  if (B == 0) return GQA_OK;
  if (!q_abs || !latent || !seq_lens || !out_lat) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(latent) || !aligned16(out_lat)) return GQA_ERR_INVALID_ARG;
  const size_t need = attn_decode_mla_absorbed_workspace_bytes(B, H, d_c, capacity);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return GQA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GQA_ERR_INVALID_ARG;
  }
  unsigned* err = error_word();
  if (!err) return GQA_ERR_CUDA;
  const float qscale = attention_scale * 1.4426950408889634f;
  float* partial = need > 0 ? static_cast<float*>(workspace) : nullptr;
  const int chunk = gqa::mla_chunk_rows(B, H, capacity);
  const cudaError_t e = gqa::launch_mla_absorbed_tc(q_abs, latent, seq_lens, out_lat, partial, B, capacity, H, d_c,
                                                    d_r, chunk, qscale, err, st, tables, mbps, bs,
                                                    num_blocks, g_withhold_first_tile);
  if (e != cudaSuccess || need == 0) return from_cuda(e);
  // the splits of each (sequence, head) merged into out_lat
  gqa::RowsParams p{};
  p.out = out_lat;
  p.partial = partial;
  p.kv_len = seq_lens;
  p.B = B;
  p.seq_q = 1;
  p.H = H;
  p.capacity = capacity;
  p.split_rows = chunk;
  p.max_splits = ceil_div(capacity, chunk);
  p.window = 0;
  p.err = err;
  return from_cuda(gqa::launch_split_combine(p, d_c, 1, st));
}

gqa_status attn_decode_mla_absorbed(const void* q_abs, const void* latent, const int32_t* seq_lens, void* out_lat,
                                    int B, int max_len, int H, int d_c, int d_r, float attention_scale, gqa_dtype dt,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || max_len <= 0 || H <= 0 || d_c <= 0 || d_r < 0 || !std::isfinite(attention_scale))
    return GQA_ERR_INVALID_ARG;
  return mla_absorbed_common(q_abs, latent, seq_lens, out_lat, B, max_len, H, d_c, d_r, attention_scale, bf16,
                             workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr, 0, 0, 0);
}

gqa_status attn_decode_mla_absorbed_paged(const void* q_abs, const void* latent_pool, const int32_t* block_tables,
                                          const int32_t* seq_lens, void* out_lat, int B, int max_blocks_per_seq,
                                          int num_blocks, int block_size, int H, int d_c, int d_r,
                                          float attention_scale, gqa_dtype dt, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0 || H <= 0 || d_c <= 0 ||
      d_r < 0 || !std::isfinite(attention_scale))
    return GQA_ERR_INVALID_ARG;
  if ((long long)max_blocks_per_seq * block_size > INT_MAX / 2) return GQA_ERR_INVALID_ARG;
  if (!gqa::mla_absorbed_paged_block_ok(block_size)) return GQA_ERR_UNSUPPORTED;
  if (B > 0 && !block_tables) return GQA_ERR_INVALID_ARG;
  return mla_absorbed_common(q_abs, latent_pool, seq_lens, out_lat, B, max_blocks_per_seq * block_size, H, d_c, d_r,
                             attention_scale, bf16, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                             block_tables, max_blocks_per_seq, block_size, num_blocks);
}

// y[b, h, :M] = W[h] x[b, h, :K] (+ the tail columns copied): the tensor-core
// kernel for the shapes it takes, else the SIMT one.
static gqa_status head_projection(const void* W, const void* x, int x_stride, void* y, int y_stride, int B, int H,
                                  int M, int K, int tail, cudaStream_t st) {
  if (gqa::head_proj_tc_supported(M, K)) {
    unsigned* err = error_word();
    if (!err) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_head_proj_tc(W, x, x_stride, y, y_stride, B, H, M, K, tail, err, st));
  }
  return from_cuda(gqa::launch_head_matvec(W, x, x_stride, y, y_stride, B, H, M, K, tail, st));
}

gqa_status mla_absorb_q(const void* q, const void* k_b, void* q_abs, int B, int H, int d_nope, int d_rope, int d_c,
                        gqa_dtype dt, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || H <= 0 || d_nope <= 0 || d_rope < 0 || d_c <= 0) return GQA_ERR_INVALID_ARG;
  if (bf16 != 1) return GQA_ERR_UNSUPPORTED;
  if (B == 0) return GQA_OK;
  if (!q || !k_b || !q_abs || q == q_abs) return GQA_ERR_INVALID_ARG;
  if (d_nope % 8 || d_rope % 8 || !aligned16(q) || !aligned16(k_b)) return GQA_ERR_INVALID_ARG;
  return head_projection(k_b, q, d_nope + d_rope, q_abs, d_c + d_rope, B, H, d_c, d_nope, d_rope,
                         static_cast<cudaStream_t>(stream));
}

gqa_status mla_unabsorb_out(const void* out_lat, const void* v_b, void* out, int B, int H, int d_c, int d_v,
                            gqa_dtype dt, void* stream) {
  const int bf16 = dtype_flag(dt);
  if (bf16 < 0 || B < 0 || H <= 0 || d_c <= 0 || d_v <= 0) return GQA_ERR_INVALID_ARG;
  if (bf16 != 1) return GQA_ERR_UNSUPPORTED;
  if (B == 0) return GQA_OK;
  if (!out_lat || !v_b || !out || out == out_lat) return GQA_ERR_INVALID_ARG;
  if (d_c % 8 || !aligned16(out_lat) || !aligned16(v_b)) return GQA_ERR_INVALID_ARG;
  return head_projection(v_b, out_lat, d_c, out, d_v, B, H, d_v, d_c, 0, static_cast<cudaStream_t>(stream));
}

gqa_status attn_get_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  unsigned word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_gqa_error_word, sizeof word) != cudaSuccess) return GQA_ERR_CUDA;
  if (word && cudaMemcpyToSymbol(g_gqa_error_word, &zero, sizeof zero) != cudaSuccess) return GQA_ERR_CUDA;
  if (word & gqa::kErrTimeout) return GQA_ERR_DEVICE_TIMEOUT;
  if (word & gqa::kErrBounds) return GQA_ERR_DEVICE_BOUNDS;
  return GQA_OK;
}

const char* gqa_status_string(gqa_status s) {
  switch (s) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported shape";
    case GQA_ERR_CUDA: return "CUDA error";
    case GQA_ERR_WORKSPACE: return "workspace missing or too small";
    case GQA_ERR_DEVICE_BOUNDS: return "device saw an index or length out of range";
    case GQA_ERR_DEVICE_TIMEOUT: return "a bounded device wait gave up";
  }
  return "unknown status";
}

int gqa_debug_withhold_first_tile(int enable) {
  const int prev = g_withhold_first_tile;
  g_withhold_first_tile = enable ? 1 : 0;
  return prev;
}

}  // extern "C"
