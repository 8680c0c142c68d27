// kernels_aux.cu -- split combine, interleaved RoPE, paged KV append, and the
// dispatch of the SIMT attention instantiations.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace gqa {

cudaError_t rows_dispatch_f32_small(const RowsParams&, int, int, int, int, cudaStream_t);
cudaError_t rows_dispatch_f32_large(const RowsParams&, int, int, int, int, cudaStream_t);
cudaError_t rows_dispatch_bf16_small(const RowsParams&, int, int, int, int, cudaStream_t);
cudaError_t rows_dispatch_bf16_d128(const RowsParams&, int, int, int, int, cudaStream_t);
cudaError_t rows_dispatch_bf16_large(const RowsParams&, int, int, int, int, cudaStream_t);

// Largest NV instantiated for these widths: at most the lanes of a row group
// (one lane per virtual head) and a register budget of ~128 floats for q and o.
int rows_max_nv(int bf16, int dk, int dv, int drot) {
  if (drot == 0 && dk == dv && dk == 16) return bf16 ? 2 : 4;
  if (drot == 0 && dk == dv && dk == 32) return bf16 ? 4 : 8;
  if (drot == 0 && dk == dv && dk == 64) return 8;
  if (drot == 0 && dk == 128 && dv == 128) return 4;
  if (drot == 0 && dk == 256 && dv == 256) return 2;
  if (dk == 192 && dv == 128 && (drot == 0 || drot == 64)) return 2;
  return 0;
}

cudaError_t launch_attn_rows_f32(const RowsParams& p, int dk, int dv, int drot, int nv, cudaStream_t st) {
  if (dk <= 64 && dk == dv) return rows_dispatch_f32_small(p, dk, dv, drot, nv, st);
  return rows_dispatch_f32_large(p, dk, dv, drot, nv, st);
}

cudaError_t launch_attn_rows_bf16(const RowsParams& p, int dk, int dv, int drot, int nv, cudaStream_t st) {
  if (dk <= 64 && dk == dv) return rows_dispatch_bf16_small(p, dk, dv, drot, nv, st);
  if (dk == 128 && dv == 128) return rows_dispatch_bf16_d128(p, dk, dv, drot, nv, st);
  return rows_dispatch_bf16_large(p, dk, dv, drot, nv, st);
}

// ---------------------------------------------------------------------------
// Split-K plan. Items are (sequence, KV head, head chunk, query-row block); an
// item with kv_hi visible keys has kv_hi / split_rows full splits and, when
// split_rows does not divide kv_hi, one partial split. The list holds every
// full split (item by item), then every partial split, so the smallest units
// come last and the tail of the dynamic schedule is short. An item whose length
// is out of range contributes one unit (split 0), on which the attention
// kernel writes its zeros. One CTA of 1024 threads.

constexpr int kPlanThreads = 1024;

// Exclusive prefix sum over the CTA; `total` receives the CTA-wide sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  total = warp_sums[(blockDim.x >> 5) - 1];
  const int before = (warp == 0 ? 0 : warp_sums[warp - 1]) + x - v;
  __syncthreads();  // warp_sums is reused by the next call
  return before;
}

// Splits of one item that hold a visible key: full ones s_first .. s_first +
// full - 1 (a window hides the splits below its lower end), then one partial
// split when split_rows does not divide the keys the last row sees.
__device__ __forceinline__ void item_split_counts(const RowsParams& p, int item, int& full, int& part,
                                                  int& s_first) {
  const int rb = item % p.n_rblocks;
  const int b = item / (p.n_rblocks * p.n_hchunks * p.Hkv);
  const int kv_len = p.kv_len ? p.kv_len[b] : (p.offsets ? p.offsets[b] : 0) + p.seq_q;
  const bool len_ok = kv_len >= p.seq_q && kv_len >= 1 && kv_len <= p.capacity;
  if (!len_ok) {
    full = 1;
    part = 0;
    s_first = 0;
    return;
  }
  const int i_last = min(rb * p.QR + p.QR, p.seq_q) - 1;
  const int kv_hi = kv_len - p.seq_q + i_last + 1;
  s_first = first_visible_key(kv_len - p.seq_q + rb * p.QR, p.window) / p.split_rows;
  full = max(0, kv_hi / p.split_rows - s_first);
  part = (kv_hi % p.split_rows) != 0;
}

// Partial units are listed longest first, in buckets of kPartBucketRows rows
// (largest-first scheduling: the last units to be taken are the shortest, so the
// CTAs run out of work at nearly the same time). The order inside a bucket is
// arbitrary; it only decides which CTA takes a unit, never what a unit computes.
constexpr int kPartBuckets = 64;

__global__ void __launch_bounds__(kPlanThreads) plan_units_kernel(const RowsParams p) {
  __shared__ int warp_sums[32];
  __shared__ int bucket_at[kPartBuckets];
  // The lengths may come from the kernel before this one (the append). The
  // attention kernel after this one may launch at once: it waits for this
  // kernel's completion before it reads the plan.
  grid_dep_wait();
  grid_dep_launch();
  const int n_items = p.B * p.Hkv * p.n_hchunks * p.n_rblocks;
  for (int i = threadIdx.x; i < kPartBuckets; i += blockDim.x) bucket_at[i] = 0;
  // thread t owns the contiguous items [lo, hi): one scan for the full units (in
  // item order), a count of the partial ones per length bucket
  const int per = (n_items + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(n_items, (int)threadIdx.x * per), hi = min(n_items, lo + per);
  auto bucket_of = [&](int item, int split) {
    const int b = item / (p.n_rblocks * p.n_hchunks * p.Hkv);
    const int rb = item % p.n_rblocks;
    const int kv_len = p.kv_len ? p.kv_len[b] : (p.offsets ? p.offsets[b] : 0) + p.seq_q;
    const int i_last = min(rb * p.QR + p.QR, p.seq_q) - 1;
    const int rows = kv_len - p.seq_q + i_last + 1 - split * p.split_rows;  // 1 .. split_rows - 1
    const int bk = (int)(((long long)(p.split_rows - rows) * kPartBuckets) / p.split_rows);
    return min(max(bk, 0), kPartBuckets - 1);  // 0: the longest
  };
  __syncthreads();
  int my_full = 0;
  for (int item = lo; item < hi; ++item) {
    int full, part, s_first;
    item_split_counts(p, item, full, part, s_first);
    my_full += full;
    if (part) atomicAdd(&bucket_at[bucket_of(item, s_first + full)], 1);
  }
  int n_full;
  int at_full = block_exclusive_scan(my_full, warp_sums, n_full);
  // bucket starts (exclusive), after the full units
  if (threadIdx.x == 0) {
    int at = n_full;
    for (int i = 0; i < kPartBuckets; ++i) {
      const int c = bucket_at[i];
      bucket_at[i] = at;
      at += c;
    }
    p.sched[1] = at;
    p.sched[0] = 0;
  }
  __syncthreads();
  for (int item = lo; item < hi; ++item) {
    int full, part, s_first;
    item_split_counts(p, item, full, part, s_first);
    for (int s = 0; s < full; ++s) p.units[at_full++] = make_int2(item, s_first + s);
    if (part) p.units[atomicAdd(&bucket_at[bucket_of(item, s_first + full)], 1)] = make_int2(item, s_first + full);
  }
}

cudaError_t launch_plan_units(const RowsParams& p, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_units_kernel, p);
}

// ---------------------------------------------------------------------------
// Split combine: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the
// splits of one (sequence, head), M = max_s m_s, in split order. Empty splits
// (m = -inf) weigh zero. One warp per output row and group of up to 256
// columns (a 512-wide row takes two warps, which read the same (m, l) pairs).

constexpr int kCombineCols = 256;  // output columns per warp

// kMaxE: output columns per lane (a warp's columns <= 32 * kMaxE <= 256).
template <typename ET, int kMaxE>
__global__ void __launch_bounds__(256) split_combine_kernel(const RowsParams p, int DV) {
  grid_dep_wait();  // the attention kernel's partials (launched as its dependent)
  const int ncg = (DV + kCombineCols - 1) / kCombineCols;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)p.B * p.seq_q * p.H * ncg) return;
  const int wid = (int)(gw / ncg);                   // the output row
  const int c0 = (int)(gw % ncg) * kCombineCols;     // its first column here
  const int DW = min(kCombineCols, DV - c0);         // columns of this warp
  const int b = wid / (p.seq_q * p.H);
  const int kv_len = p.kv_len ? p.kv_len[b] : (p.offsets ? p.offsets[b] : 0) + p.seq_q;
  if (!(kv_len >= p.seq_q && kv_len >= 1 && kv_len <= p.capacity)) return;  // attention wrote zeros
  // seq_q == 1 whenever splitting: the row sits at kv_len - 1
  const int n = (kv_len + p.split_rows - 1) / p.split_rows;
  const int s_lo = first_visible_key(kv_len - 1, p.window) / p.split_rows;  // splits below the window hold no key
  if (n - s_lo <= 1) return;  // attention wrote the output itself
  const int stride = DV + 2;
  const float* P = p.partial + (size_t)wid * p.max_splits * stride;
  // the sink logit (log2 domain) joins the denominator once per row and head
  const float z2 = p.sinks ? __ldg(p.sinks + wid % p.H) * kLog2e : -INFINITY;
  ET* out = reinterpret_cast<ET*>(p.out) + (size_t)wid * DV + c0;
  // Few splits (the common case): every load of the row is issued at once --
  // each split's (m, l) and this lane's column pairs d = 2 lane + 64 e of its
  // o (8-byte aligned: rows of d_v + 2 floats, d_v and c0 even) -- so the row
  // costs one round trip; the weights and sums then run in split order as
  // below, and the output is stored as pairs. At most 16 partial values per lane.
  constexpr int kFast = 16 / kMaxE;
  if (n - s_lo <= kFast && (DV & 1) == 0) {
    const int nk = n - s_lo;
    float2 v[kFast][kMaxE / 2];
    float mk[kFast], lk[kFast];
#pragma unroll
    for (int j = 0; j < kFast; ++j) {
      const bool ok = j < nk;
      const float* row = P + (size_t)(s_lo + (ok ? j : 0)) * stride;
      mk[j] = ok ? __ldcg(row) : -INFINITY;
      lk[j] = ok ? __ldcg(row + 1) : 0.f;
#pragma unroll
      for (int e = 0; e < kMaxE / 2; ++e) {
        const int d = 2 * lane + 64 * e;
        v[j][e] = (ok && d < DW) ? __ldcg(reinterpret_cast<const float2*>(row + 2 + c0 + d)) : make_float2(0.f, 0.f);
      }
    }
    float M = z2;
#pragma unroll
    for (int j = 0; j < kFast; ++j) M = fmaxf(M, mk[j]);
    float2 acc[kMaxE / 2];
#pragma unroll
    for (int e = 0; e < kMaxE / 2; ++e) acc[e] = make_float2(0.f, 0.f);
    float dsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int j = 0; j < kFast; ++j) {
        const float w = (mk[j] == -INFINITY) ? 0.f : exp2f(mk[j] - M);
        dsum = fmaf(w, lk[j], dsum);
#pragma unroll
        for (int e = 0; e < kMaxE / 2; ++e) {
          acc[e].x = fmaf(w, v[j][e].x, acc[e].x);
          acc[e].y = fmaf(w, v[j][e].y, acc[e].y);
        }
      }
    }
    const float den = M == -INFINITY ? 0.f : (p.sinks ? exp2f(z2 - M) : 0.f) + dsum;
#pragma unroll
    for (int e = 0; e < kMaxE / 2; ++e) {
      const int d = 2 * lane + 64 * e;
      if (d >= DW) continue;
      const float a = den > 0.f ? acc[e].x / den : 0.f, c = den > 0.f ? acc[e].y / den : 0.f;
      if constexpr (sizeof(ET) == 2)
        *reinterpret_cast<__nv_bfloat162*>(out + d) = __floats2bfloat162_rn(a, c);
      else
        *reinterpret_cast<float2*>(out + d) = make_float2(a, c);
    }
    return;
  }
  float M = z2;
  for (int s = s_lo + lane; s < n; s += 32) M = fmaxf(M, P[(size_t)s * stride]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (M == -INFINITY) {
    for (int d = lane; d < DW; d += 32) out[d] = Elem<ET>::from_f32(0.f);
    return;
  }
  // Each split's weight once (lane s % 32 holds split s's), the weighted row sums
  // reduced in a fixed butterfly order; every lane then walks the splits in order,
  // the weight broadcast, its output columns d = lane + 32 e read as coalesced rows.
  float acc[kMaxE];
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) acc[e] = 0.f;
  float den_part = 0.f;
  for (int s0 = s_lo; s0 < n; s0 += 32) {
    const int s = s0 + lane;
    float w = 0.f;
    if (s < n) {
      const float ms = P[(size_t)s * stride];
      w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      den_part = fmaf(w, P[(size_t)s * stride + 1], den_part);
    }
    // The rows of up to kBatch splits are loaded before any of them is
    // accumulated, so that many loads are in flight per lane; the sum still
    // runs over the splits in order.
    constexpr int kBatch = 16 / kMaxE;
    const int cnt = min(32, n - s0);
    for (int j0 = 0; j0 < cnt; j0 += kBatch) {
      float v[kBatch][kMaxE];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const float* row = P + (size_t)(s0 + j0 + jj) * stride + 2 + c0;
#pragma unroll
        for (int e = 0; e < kMaxE; ++e)
          v[jj][e] = (j0 + jj < cnt && lane + 32 * e < DW) ? __ldcg(row + lane + 32 * e) : 0.f;
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const float wj = __shfl_sync(0xffffffffu, w, (j0 + jj) & 31);
        if (j0 + jj < cnt) {
#pragma unroll
          for (int e = 0; e < kMaxE; ++e)
            if (lane + 32 * e < DW) acc[e] = fmaf(wj, v[jj][e], acc[e]);
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) den_part += __shfl_xor_sync(0xffffffffu, den_part, off);
  const float den = (p.sinks ? exp2f(z2 - M) : 0.f) + den_part;
#pragma unroll
  for (int e = 0; e < kMaxE; ++e)
    if (lane + 32 * e < DW) out[lane + 32 * e] = Elem<ET>::from_f32(den > 0.f ? acc[e] / den : 0.f);
}

cudaError_t launch_split_combine(const RowsParams& p, int dv, int bf16, cudaStream_t st) {
  // d_v up to 512 (the latent width of the absorbed MLA decode): a warp per row
  // and group of up to 256 columns, in lanes' shares of 4 or 8 columns.
  if (dv > 512) return cudaErrorNotSupported;
  const long long warps = (long long)p.B * p.seq_q * p.H * ((dv + kCombineCols - 1) / kCombineCols);
  if (warps <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  const long long blocks = (warps + warps_per_block - 1) / warps_per_block;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  // Launched as a programmatic dependent of the attention kernel before it:
  // its CTAs may start while that kernel finishes, and wait for it
  // (grid_dep_wait) before reading the partials.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(32 * warps_per_block);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) {
    if (dv <= 128) return cudaLaunchKernelEx(&cfg, split_combine_kernel<__nv_bfloat16, 4>, p, dv);
    return cudaLaunchKernelEx(&cfg, split_combine_kernel<__nv_bfloat16, 8>, p, dv);
  }
  if (dv <= 128) return cudaLaunchKernelEx(&cfg, split_combine_kernel<float, 4>, p, dv);
  return cudaLaunchKernelEx(&cfg, split_combine_kernel<float, 8>, p, dv);
}

// ---------------------------------------------------------------------------
// Interleaved RoPE. The angle pos * theta^(-2t/rot_dim) has to be reduced
// modulo 2*pi accurately (positions reach 32k, where a plain fp32 angle would
// be off by ~2e-3 rad); sine and cosine of the reduced angle come from the
// fp32 sincosf, the rotation is done in fp32 and rounded once on store.

// 2*pi split into a double and the double nearest to its remainder (Cody and
// Waite's reduction): a - n*HI - n*LO keeps ~1e-15 rad for |n| < 2^20.
constexpr double kTwoPiHi = 6.283185307179586;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189535;

__device__ __forceinline__ void rope_cos_sin(double pos, double w, float* c, float* s) {
  const double a = pos * w;
  const double n = rint(a * kInvTwoPi);
  const double r = fma(-n, kTwoPiLo, fma(-n, kTwoPiHi, a));
  sincosf((float)r, s, c);
}

// The same in fp32 arithmetic, which this GPU runs far faster than fp64, for
// |pos| < 2^24 (the position exact in a float). The frequency comes as a float
// pair w_hi + w_lo within 2^-48 of the double; the product pos * w is formed
// without error in a_hi + e (Dekker and Kahan's two-product: one FMA gives the
// rounding error of pos * w_hi), and the reduction modulo 2*pi is Cody and
// Waite's with 2*pi as the sum of three floats, one FMA per part. The reduced
// angle is within ~3e-7 rad of the exact one (the fp64 form, which also rounds
// it to a float before sincosf, within ~1.2e-7).
constexpr float kTwoPiF1 = 6.2831854820251465f;       // the float nearest 2*pi
constexpr float kTwoPiF2 = -1.7484555314695172e-07f;  // ... nearest 2*pi - kTwoPiF1
constexpr float kTwoPiF3 = -6.8604980400235275e-15f;  // ... nearest what remains (4e-23 left)
constexpr float kInvTwoPiF = 0.15915493667125702f;

__device__ __forceinline__ void rope_cos_sin_f(int pos, float w_hi, float w_lo, double w, float* c, float* s) {
  if (pos >= (1 << 24) || pos <= -(1 << 24)) {  // not exact as a float
    rope_cos_sin((double)pos, w, c, s);
    return;
  }
  const float p = (float)pos;
  const float a_hi = p * w_hi;
  const float a_lo = fmaf(p, w_lo, fmaf(p, w_hi, -a_hi));  // the rounding error of p * w_hi, plus p * w_lo
  const float n = rintf(a_hi * kInvTwoPiF);
  float r = fmaf(-n, kTwoPiF1, a_hi);
  r = fmaf(-n, kTwoPiF2, r);
  r = fmaf(-n, kTwoPiF3, r);
  sincosf(r + a_lo, s, c);
}

// The rot_dim/2 frequencies theta^(-2t/rot_dim), t < rot_dim/2, computed once
// per call on the host in double (w) and split into a float pair (w_hi + w_lo),
// passed by value (they depend only on the call's scalar arguments).
struct RopeFreqs {
  double w[128];
  float w_hi[128], w_lo[128];
};

RopeFreqs rope_freqs(int rot_dim, double theta) {
  RopeFreqs f{};
  for (int t = 0; t < rot_dim / 2 && t < 128; ++t) {
    f.w[t] = std::pow(theta, -2.0 * t / rot_dim);
    f.w_hi[t] = (float)f.w[t];
    f.w_lo[t] = (float)(f.w[t] - (double)f.w_hi[t]);
  }
  return f;
}

template <typename ET>
__device__ __forceinline__ void rotate_pair(ET* x, float c, float s) {
  const float x0 = Elem<ET>::to_f32(x[0]), x1 = Elem<ET>::to_f32(x[1]);
  x[0] = Elem<ET>::from_f32(fmaf(x0, c, -x1 * s));
  x[1] = Elem<ET>::from_f32(fmaf(x0, s, x1 * c));
}

// A pair (x[2t], x[2t+1]) as one 4-byte (bf16) or 8-byte (f32) access: the
// element offset of a pair is even and tensors are 16-byte aligned.
template <typename ET>
struct Pair;
template <>
struct Pair<__nv_bfloat16> {
  static __device__ __forceinline__ float2 load(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
  }
};
template <>
struct Pair<float> {
  static __device__ __forceinline__ float2 load(const float* p) { return *reinterpret_cast<const float2*>(p); }
  static __device__ __forceinline__ void store(float* p, float a, float b) {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
  }
};

// One thread per (token, pair): the angle once, then the pair of every head,
// sixteen heads' loads in flight at a time (all of them for up to 16 heads),
// so that a thread waits on memory once per sixteen heads; with a second
// tensor of the same tokens (the keys beside the queries), its heads' pairs
// next, turned by the same angle.
constexpr int kRopeHeadsInFlight = 16;
constexpr int kRopeHeadsInFlight2 = 4;  // of the second tensor (the k heads of a GQA pair)

template <typename ET>
__global__ void __launch_bounds__(128) rope_kernel(ET* x, const int32_t* positions, int B, int T, int heads, int d,
                                                   int heads_outer, int rot_offset, int rot_dim, const RopeFreqs fr,
                                                   ET* x2, int heads2, int heads_outer2) {
  const int npairs = rot_dim / 2;
  // The frequencies into shared memory first: read from the parameter space at
  // a different index in every lane, each warp's load would be serialised.
  __shared__ double w_s[128];
  __shared__ float2 wf_s[128];
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
    w_s[i] = fr.w[i];
    wf_s[i] = make_float2(fr.w_hi[i], fr.w_lo[i]);
  }
  // launched as a programmatic dependent: x and the positions may come from the
  // kernel before this one; the next launch may start setting up at once
  grid_dep_wait();
  grid_dep_launch();
  __syncthreads();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)B * T * npairs) return;
  const int pr = (int)(idx % npairs);
  const long long tok = idx / npairs;  // b * T + t
  const int b = (int)(tok / T), t = (int)(tok % T);
  const int pos = positions[tok];
  // head h's pair at p0 + h * hstride ([B, T, heads, d] or, heads outer, [B, heads, T, d])
  const size_t hstride = heads_outer ? (size_t)T * d : (size_t)d;
  ET* p0 = x + (heads_outer ? ((size_t)b * heads * T + t) : (size_t)tok * heads) * d + rot_offset + 2 * pr;
  // a second tensor of the same tokens (x2 != NULL) turns by the same angle
  const size_t hstride2 = heads_outer2 ? (size_t)T * d : (size_t)d;
  ET* p2 = x2 ? x2 + (heads_outer2 ? ((size_t)b * heads2 * T + t) : (size_t)tok * heads2) * d + rot_offset + 2 * pr
              : nullptr;
  // the first heads' pairs (of both tensors) are requested before the angle
  // waits on the position
  float2 xv[kRopeHeadsInFlight], xv2[kRopeHeadsInFlight2];
#pragma unroll
  for (int u = 0; u < kRopeHeadsInFlight; ++u)
    if (u < heads) xv[u] = Pair<ET>::load(p0 + (size_t)u * hstride);
#pragma unroll
  for (int u = 0; u < kRopeHeadsInFlight2; ++u)
    if (p2 && u < heads2) xv2[u] = Pair<ET>::load(p2 + (size_t)u * hstride2);
  float c, s;
  rope_cos_sin_f(pos, wf_s[pr].x, wf_s[pr].y, w_s[pr], &c, &s);
  for (int h0 = 0; h0 < heads; h0 += kRopeHeadsInFlight) {
    if (h0 > 0) {
#pragma unroll
      for (int u = 0; u < kRopeHeadsInFlight; ++u)
        if (h0 + u < heads) xv[u] = Pair<ET>::load(p0 + (size_t)(h0 + u) * hstride);
    }
#pragma unroll
    for (int u = 0; u < kRopeHeadsInFlight; ++u)
      if (h0 + u < heads)
        Pair<ET>::store(p0 + (size_t)(h0 + u) * hstride, fmaf(xv[u].x, c, -xv[u].y * s),
                        fmaf(xv[u].x, s, xv[u].y * c));
  }
  if (!p2) return;
  for (int h0 = 0; h0 < heads2; h0 += kRopeHeadsInFlight2) {
    if (h0 > 0) {
#pragma unroll
      for (int u = 0; u < kRopeHeadsInFlight2; ++u)
        if (h0 + u < heads2) xv2[u] = Pair<ET>::load(p2 + (size_t)(h0 + u) * hstride2);
    }
#pragma unroll
    for (int u = 0; u < kRopeHeadsInFlight2; ++u)
      if (h0 + u < heads2)
        Pair<ET>::store(p2 + (size_t)(h0 + u) * hstride2, fmaf(xv2[u].x, c, -xv2[u].y * s),
                        fmaf(xv2[u].x, s, xv2[u].y * c));
  }
}

cudaError_t launch_rope(void* x, const int32_t* positions, int B, int T, int heads, int d, int heads_outer,
                        int rot_offset, int rot_dim, double theta, int bf16, cudaStream_t st, void* x2, int heads2,
                        int heads_outer2) {
  const long long total = (long long)B * T * (rot_dim / 2);
  if (total <= 0 || heads <= 0) return cudaSuccess;
  if (rot_dim > 256) return cudaErrorNotSupported;
  const unsigned blocks = (unsigned)((total + 127) / 128);
  const RopeFreqs fr = rope_freqs(rot_dim, theta);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16)
    return cudaLaunchKernelEx(&cfg, rope_kernel<__nv_bfloat16>, reinterpret_cast<__nv_bfloat16*>(x), positions, B, T,
                              heads, d, heads_outer, rot_offset, rot_dim, fr, reinterpret_cast<__nv_bfloat16*>(x2),
                              heads2, heads_outer2);
  return cudaLaunchKernelEx(&cfg, rope_kernel<float>, reinterpret_cast<float*>(x), positions, B, T, heads, d,
                            heads_outer, rot_offset, rot_dim, fr, reinterpret_cast<float*>(x2), heads2, heads_outer2);
}

// ---------------------------------------------------------------------------
// Paged append of one row per sequence (one CTA per sequence): position
// p = lens_in[b] is read before anything is written; q (all heads) and the new
// k (all KV heads) are rotated at p; k and v go to slot p % bs of block
// tables[b][p / bs]; lens_out[b] = p + 1.

template <typename ET>
__global__ void __launch_bounds__(128) append_kernel(ET* q, const ET* k_new, const ET* v_new, ET* k_pool, ET* v_pool,
                                                     const int32_t* tables, const int32_t* lens_in, int32_t* lens_out,
                                                     int mbps, int num_blocks, int bs, int H, int Hkv, int dk, int dv,
                                                     bool rope, const RopeFreqs fr, int rot_offset, int rot_dim,
                                                     unsigned* err) {
  const int b = blockIdx.x;
  // launched as a programmatic dependent: the lengths and the rows may come from
  // the kernel before this one; the next launch (the unit plan) may start at once
  grid_dep_wait();
  grid_dep_launch();
  const int p = lens_in[b];
  const bool pos_ok = p >= 0 && (long long)p < (long long)mbps * bs;
  const int blk = pos_ok ? tables[(size_t)b * mbps + p / bs] : -1;
  const bool ok = pos_ok && blk >= 0 && blk < num_blocks;
  __syncthreads();  // every thread has read lens_in[b] (lens_out may alias it)
  if (!ok) {
    if (threadIdx.x == 0) {
      raise_error(err, kErrBounds);
      lens_out[b] = p;
    }
    return;
  }
  const int row = p % bs;
  // Vector path: q, k and v in 16-byte chunks (whole rotary pairs: a chunk lies
  // wholly inside or outside the rotated columns), each pair's (cos, sin) at p
  // computed once and shared; every chunk's load of a round issued before any
  // rotation or store, so a thread waits on memory once per round (one element
  // or pair at a time, the loads and stores of a CTA had been ~50 round trips).
  constexpr int V = Elem<ET>::kPerChunk;
  const bool vec = dk % V == 0 && dv % V == 0 && (!rope || (rot_offset % V == 0 && rot_dim % V == 0)) &&
                   ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_new) |
                     reinterpret_cast<uintptr_t>(v_new) | reinterpret_cast<uintptr_t>(k_pool) |
                     reinterpret_cast<uintptr_t>(v_pool)) & 15) == 0;
  if (vec) {
    __shared__ float2 cs[128];  // (cos, sin) of rotary pair t at p
    if (rope)
      for (int pr = threadIdx.x; pr < rot_dim / 2; pr += blockDim.x) rope_cos_sin((double)p, fr.w[pr], &cs[pr].x, &cs[pr].y);
    __syncthreads();
    const int cpk = dk / V, cpv = dv / V;  // chunks per row
    const int nq = H * cpk, nk = Hkv * cpk, nv = Hkv * cpv, n = nq + nk + nv;
    // chunk i: (source, destination, first rotated pair or -1)
    auto chunk = [&](int i, const ET*& src, ET*& dst, int& t0) {
      t0 = -1;
      int c0;
      if (i < nq) {
        const int h = i / cpk;
        c0 = (i % cpk) * V;
        src = dst = q + ((size_t)b * H + h) * dk + c0;
      } else if (i < nq + nk) {
        const int kh = (i - nq) / cpk;
        c0 = ((i - nq) % cpk) * V;
        src = k_new + ((size_t)b * Hkv + kh) * dk + c0;
        dst = k_pool + (((size_t)blk * Hkv + kh) * bs + row) * dk + c0;
      } else {
        const int kh = (i - nq - nk) / cpv;
        src = v_new + ((size_t)b * Hkv + kh) * dv + ((i - nq - nk) % cpv) * V;
        dst = v_pool + (((size_t)blk * Hkv + kh) * bs + row) * dv + ((i - nq - nk) % cpv) * V;
        return;
      }
      if (rope && c0 >= rot_offset && c0 < rot_offset + rot_dim) t0 = (c0 - rot_offset) / 2;
    };
    constexpr int kRound = 8;  // chunks per thread in flight
    for (int i0 = threadIdx.x; i0 < n; i0 += kRound * blockDim.x) {
      uint4 v[kRound];
#pragma unroll
      for (int u = 0; u < kRound; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        if (i >= n) continue;
        const ET* src;
        ET* dst;
        int t0;
        chunk(i, src, dst, t0);
        v[u] = *reinterpret_cast<const uint4*>(src);
      }
#pragma unroll
      for (int u = 0; u < kRound; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        if (i >= n) continue;
        const ET* src;
        ET* dst;
        int t0;
        chunk(i, src, dst, t0);
        if (t0 >= 0) {  // rotate the chunk's V / 2 pairs as rotate_pair does
          ET* e = reinterpret_cast<ET*>(&v[u]);
#pragma unroll
          for (int j = 0; j < V / 2; ++j) {
            const float2 w = cs[t0 + j];
            const float x0 = Elem<ET>::to_f32(e[2 * j]), x1 = Elem<ET>::to_f32(e[2 * j + 1]);
            e[2 * j] = Elem<ET>::from_f32(fmaf(x0, w.x, -x1 * w.y));
            e[2 * j + 1] = Elem<ET>::from_f32(fmaf(x0, w.y, x1 * w.x));
          }
        }
        *reinterpret_cast<uint4*>(dst) = v[u];
      }
    }
  } else {
    if (rope) {
      for (int pr = threadIdx.x; pr < rot_dim / 2; pr += blockDim.x) {
        float c, s;
        rope_cos_sin((double)p, fr.w[pr], &c, &s);
        const int e = rot_offset + 2 * pr;
        for (int h = 0; h < H; ++h) rotate_pair(q + ((size_t)b * H + h) * dk + e, c, s);
        for (int kh = 0; kh < Hkv; ++kh) {
          ET pair[2] = {k_new[((size_t)b * Hkv + kh) * dk + e], k_new[((size_t)b * Hkv + kh) * dk + e + 1]};
          rotate_pair(pair, c, s);
          ET* dst = k_pool + (((size_t)blk * Hkv + kh) * bs + row) * dk + e;
          dst[0] = pair[0];
          dst[1] = pair[1];
        }
      }
    }
    for (int idx = threadIdx.x; idx < Hkv * dk; idx += blockDim.x) {
      const int kh = idx / dk, e = idx % dk;
      if (rope && e >= rot_offset && e < rot_offset + rot_dim) continue;  // written rotated above
      k_pool[(((size_t)blk * Hkv + kh) * bs + row) * dk + e] = k_new[((size_t)b * Hkv + kh) * dk + e];
    }
    for (int idx = threadIdx.x; idx < Hkv * dv; idx += blockDim.x) {
      const int kh = idx / dv, e = idx % dv;
      v_pool[(((size_t)blk * Hkv + kh) * bs + row) * dv + e] = v_new[((size_t)b * Hkv + kh) * dv + e];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) lens_out[b] = p + 1;
}

cudaError_t launch_append(void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                          const int32_t* tables, const int32_t* lens_in, int32_t* lens_out, int B, int mbps,
                          int num_blocks, int bs, int H, int Hkv, int dk, int dv, double theta, int rot_offset,
                          int rot_dim, int bf16, unsigned* err, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  const bool rope = theta > 0.0 && rot_dim > 0;
  if (rope && rot_dim > 256) return cudaErrorNotSupported;
  const RopeFreqs fr = rope_freqs(rope ? rot_dim : 0, theta);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16)
    return cudaLaunchKernelEx(&cfg, append_kernel<__nv_bfloat16>, reinterpret_cast<__nv_bfloat16*>(q),
                              reinterpret_cast<const __nv_bfloat16*>(k_new), reinterpret_cast<const __nv_bfloat16*>(v_new),
                              reinterpret_cast<__nv_bfloat16*>(k_pool), reinterpret_cast<__nv_bfloat16*>(v_pool), tables,
                              lens_in, lens_out, mbps, num_blocks, bs, H, Hkv, dk, dv, rope, fr, rot_offset, rot_dim,
                              err);
  return cudaLaunchKernelEx(&cfg, append_kernel<float>, reinterpret_cast<float*>(q), reinterpret_cast<const float*>(k_new),
                            reinterpret_cast<const float*>(v_new), reinterpret_cast<float*>(k_pool),
                            reinterpret_cast<float*>(v_pool), tables, lens_in, lens_out, mbps, num_blocks, bs, H, Hkv,
                            dk, dv, rope, fr, rot_offset, rot_dim, err);
}

}  // namespace gqa
