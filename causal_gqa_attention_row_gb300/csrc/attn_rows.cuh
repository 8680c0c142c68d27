// attn_rows.cuh -- SIMT split-K attention of query rows against a KV cache.
//
// The operation (kopitiam-runtime src/attention.rs, `attention_forward`,
// `causal_mask`, `repeat_kv_heads`): query head h reads KV head h / G; query row
// i at position offset + i sees keys 0..=offset + i; softmax over the visible
// keys of scale * q.k, then the weighted sum of V.
//
// One CTA is one work item: (sequence b, KV head kvh, a chunk of GH of that KV
// head's G query heads, a block of QR query rows, a split of the key range).
// Its GH*QR = NV "virtual heads" (query row, query head) all read the SAME K/V
// rows, so each K/V row crosses HBM once per KV head however large the group
// (frink-models src/decoder/attn_block.rs and kopitiam's module doc: every
// query head of a group genuinely shares its KV head).
//
// Data path: one producer warp streams K/V tiles of T rows into an NS-deep
// shared-memory ring with 1-D bulk copies (cp.async.bulk, the TMA engine)
// completing on mbarriers. Contiguous caches need one copy per tile and
// operand; paged caches one per block segment, the block-table gather done by
// the copy engine (frink-models src/decoder/attn_block.rs, `push_and_attend_row`,
// paged arm). Four compute warps consume the ring.
//
// Compute mapping: a "row group" of L lanes owns one key row at a time; lane li
// holds the 16-byte chunks li, li+L, li+2L, ... of q (fp32, pre-scaled by
// scale*log2 e) for each virtual head and of its own output accumulators, as
// float2 pairs for the paired FFMA2 instruction. A row's NV scores are L-lane
// partial dot products finished by a halving ("transpose") butterfly: each
// shuffle step also halves the number of heads a lane carries, so the lane ends
// up owning ONE head's full score. That lane alone runs the online softmax of
// its head (reference max m, denominator l) and the probability p is broadcast
// to the group with one shuffle per head.
//
// Each row group takes the 2 rows it owns in a tile as one chunk: two
// independent dot products, one max/rescale check, two exponentials. Rescaling
// is lazy: o and l move to a new reference max only when a score exceeds the
// current one by more than 2^8, which keeps every term <= 256 and leaves o / l
// unchanged. At the end the row groups are merged through shared memory in a
// fixed order (log-sum-exp), then written as the output (one split) or as a
// partial (m, l, o) that the combine kernel merges, again in a fixed order.
//
// Determinism: split boundaries are multiples of kSplitRows, tiles multiples of
// T rows from the split start, and the row -> row-group assignment a function of
// the key index only. The arithmetic on a key row therefore does not depend on
// where the row lives (contiguous or paged), on the block table, or on the other
// sequences of the batch: paged and contiguous results are bit-identical.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace gqa {

constexpr int kRowsWarps = 4;  // compute warps
constexpr int kRowsThreads = (kRowsWarps + 1) * 32;
constexpr int kMaxStages = 4;
constexpr int kRingBudget = 128 * 1024;  // shared-memory ring per CTA (two CTAs per SM)
constexpr float kRescaleLog2 = 8.0f;

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int clog2(int x) { return x <= 1 ? 0 : 1 + clog2(x / 2); }

template <typename ET, int DK, int DV, int DROT, int NV>
struct RowsCfg {
  static constexpr int CH = Elem<ET>::kPerChunk;
  static constexpr int ES = (int)sizeof(ET);
  static constexpr int DN = DK - DROT;  // key part stored per KV head
  static constexpr int KCH = DK / CH, VCH = DV / CH, NCH = DN / CH;
  static constexpr int L = cmin(8, cmin(KCH, VCH));  // lanes per row group
  static constexpr int QK = KCH / L, QV = VCH / L;   // chunks per lane
  static constexpr int EK = QK * CH, EV = QV * CH;   // elements per lane
  static constexpr int RGW = 32 / L;                 // row groups per warp
  static constexpr int NRG = kRowsWarps * RGW;
  static constexpr int T = 2 * NRG;                  // rows per tile: two per row group
  static constexpr int kN = T * DN * ES, kR = T * DROT * ES, kV = T * DV * ES;
  static constexpr int stage_bytes = kN + kR + kV;
  static constexpr int row_bytes = (DN + DROT + DV) * ES;
  static constexpr int NS = cmax(2, cmin(kMaxStages, kRingBudget / stage_bytes));  // ring depth
  static constexpr int merge_bytes = NRG * NV * (DV + 2) * 4;
  static constexpr int data_bytes = cmax(NS * stage_bytes, merge_bytes);
  static constexpr int kHeader = 128;  // mbarriers + flags
  static constexpr int smem_bytes = kHeader + data_bytes;
  static constexpr int MIN_CTAS = 2;  // CTAs per SM the register budget targets
  static_assert(DK % CH == 0 && DV % CH == 0 && DN % CH == 0, "head widths must be whole 16-byte chunks");
  static_assert(KCH % L == 0 && VCH % L == 0 && NCH % L == 0, "chunks must split evenly over a row group");
  static_assert(32 % L == 0, "row groups must tile a warp");
  static_assert(NV <= L, "a row group needs at least one lane per virtual head");
  static_assert(kSplitRows % T == 0, "split boundaries must fall on tile boundaries");
};

// Head owned by lane li of a row group after the halving butterfly: at the
// step with offset L >> (k+1) the lanes with that bit set keep the upper half
// of the heads they carried.
template <int NV, int L>
__device__ __forceinline__ int owned_head(int li) {
  int h = 0;
#pragma unroll
  for (int k = 0, n = NV; n > 1; ++k, n >>= 1)
    if (li & (L >> (k + 1))) h += n >> 1;
  return h;
}

// Lowest lane of a row group that owns head h (inverse of owned_head).
template <int NV, int L>
__host__ __device__ constexpr int owner_lane(int h) {
  int li = 0;
  for (int k = 0, n = NV; n > 1; ++k, n >>= 1)
    if (h & (n >> 1)) li |= L >> (k + 1);
  return li;
}

// Sum NV per-lane partial scores over the L lanes of a row group; each lane
// returns the full score of its owned head.
template <int NV, int L>
__device__ __forceinline__ float reduce_own(const float (&v)[NV], int li) {
  float cur[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) cur[i] = v[i];
  int off = L >> 1;
#pragma unroll
  for (int n = NV; n > 1; n >>= 1) {
    const bool upper = (li & off) != 0;
    const int half = n >> 1;
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
      if (i < half) {
        const float keep = upper ? cur[i + half] : cur[i];
        const float send = upper ? cur[i] : cur[i + half];
        cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    off >>= 1;
  }
  float s = cur[0];
#pragma unroll
  for (; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

// 2^x on the special-function unit (the PTX ex2.approx instruction, flushing
// subnormal results to zero; exp2(-inf) = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename ET>
__device__ __forceinline__ void chunk_to_f2(const uint4 u, float2* f);

template <>
__device__ __forceinline__ void chunk_to_f2<__nv_bfloat16>(const uint4 u, float2* f) {
  f[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
  f[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  f[2] = make_float2(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u));
  f[3] = make_float2(__uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
}

template <>
__device__ __forceinline__ void chunk_to_f2<float>(const uint4 u, float2* f) {
  f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
  f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
}

// Warp-uniform bounded wait. On a timeout (or an abort raised elsewhere in the
// CTA) every lane returns false and the abort flag and error word are set.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* err) {
  bool ok = (*abort_flag == 0) && mbar_wait(bar, parity);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) {
    *abort_flag = 1;
    raise_error(err, kErrTimeout);
  }
  return ok;
}

template <typename ET, int DK, int DV, int DROT, int NV>
__global__ void __launch_bounds__(kRowsThreads, RowsCfg<ET, DK, DV, DROT, NV>::MIN_CTAS)
    attn_rows_kernel(const RowsParams p) {
  using C = RowsCfg<ET, DK, DV, DROT, NV>;
  constexpr int CH = C::CH, L = C::L, T = C::T, kStages = C::NS;
  constexpr int H2K = C::EK / 2, H2V = C::EV / 2;  // float2 pairs per lane
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
  volatile int* bad_table = abort_flag + 1;
  unsigned char* data = smem + C::kHeader;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the work item
  const int split = blockIdx.y;
  int item = blockIdx.x;
  const int rb = item % p.n_rblocks;
  item /= p.n_rblocks;
  const int hc = item % p.n_hchunks;
  item /= p.n_hchunks;
  const int kvh = item % p.Hkv;
  const int b = item / p.Hkv;

  const int kv_len = p.kv_len ? p.kv_len[b] : (p.offsets ? p.offsets[b] : 0) + p.seq_q;
  const int i0 = rb * p.QR;
  const int i_last = min(i0 + p.QR, p.seq_q) - 1;
  const bool len_ok = kv_len >= p.seq_q && kv_len >= 1 && kv_len <= p.capacity;
  const int kv_hi = len_ok ? kv_len - p.seq_q + i_last + 1 : 0;  // keys the last row sees
  const int nsplit = (kv_hi + p.split_rows - 1) / p.split_rows;
  const int r0 = split * p.split_rows;
  const int r1 = min(r0 + p.split_rows, kv_hi);

  if (!len_ok) {
    // Length out of range: record it, write zeros once, touch no K/V.
    if (split == 0) {
      if (threadIdx.x == 0 && kvh == 0 && hc == 0 && rb == 0) raise_error(p.err, kErrBounds);
      for (int idx = threadIdx.x; idx < NV * DV; idx += blockDim.x) {
        const int vh = idx / DV, d = idx % DV;
        const int iq = i0 + vh / p.GH;
        if (iq >= p.seq_q) continue;
        const int h = kvh * p.G + hc * p.GH + vh % p.GH;
        reinterpret_cast<ET*>(p.out)[(((size_t)b * p.seq_q + iq) * p.H + h) * DV + d] = Elem<ET>::from_f32(0.f);
      }
    }
    return;
  }
  if (r0 >= r1) return;  // this split lies past the last visible key

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kRowsWarps);
    }
    *abort_flag = 0;
    *bad_table = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // ---- paged: check every block-table entry this item reads before any copy
  if (p.paged) {
    const int blk0 = r0 / p.bs, blk1 = (r1 - 1) / p.bs;
    for (int bi = blk0 + (int)threadIdx.x; bi <= blk1; bi += blockDim.x) {
      const int e = p.tables[(size_t)b * p.mbps + bi];
      if (e < 0 || e >= p.num_blocks) *bad_table = 1;
    }
    __syncthreads();
    if (*bad_table) {
      if (threadIdx.x == 0) raise_error(p.err, kErrBounds);
      // An empty partial (m = -inf, l = 0) or zeros: no K/V row is read.
      for (int idx = threadIdx.x; idx < NV * DV; idx += blockDim.x) {
        const int vh = idx / DV, d = idx % DV;
        const int iq = i0 + vh / p.GH;
        if (iq >= p.seq_q) continue;
        const int h = kvh * p.G + hc * p.GH + vh % p.GH;
        const size_t row = ((size_t)b * p.seq_q + iq) * p.H + h;
        if (nsplit == 1) {
          reinterpret_cast<ET*>(p.out)[row * DV + d] = Elem<ET>::from_f32(0.f);
        } else {
          float* P = p.partial + (row * p.max_splits + split) * (DV + 2);
          if (d == 0) {
            P[0] = -INFINITY;
            P[1] = 0.f;
          }
          P[2 + d] = 0.f;
        }
      }
      return;
    }
  }

  const int ntiles = (r1 - r0 + T - 1) / T;
  const int rgw = lane / L, li = lane % L;
  const int own = owned_head<NV, L>(li);  // the virtual head whose softmax this lane runs

  // output accumulators (all heads, this lane's chunks) and the owned head's state
  float2 o2[NV][H2V];
#pragma unroll
  for (int vh = 0; vh < NV; ++vh)
#pragma unroll
    for (int e = 0; e < H2V; ++e) o2[vh][e] = make_float2(0.f, 0.f);
  float m_ref = -INFINITY, l_sum = 0.f;

  if (warp == kRowsWarps) {
    // ================= producer warp =================
    const uint64_t pol = l2_policy_evict_first();
    int last_issued[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) last_issued[s] = -1;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % kStages;
      if (t >= kStages) {
        bool ok = true;
        if (lane == 0) ok = (*abort_flag == 0) && mbar_wait(&empty[s], ((t / kStages) - 1) & 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) {
            *abort_flag = 1;
            raise_error(p.err, kErrTimeout);
          }
          break;
        }
      }
      if (*abort_flag) break;
      const int tr0 = r0 + t * T;
      const int n = min(T, r1 - tr0);
      if (p.debug_withhold && t == 0) continue;  // test hook: this tile never arrives
#pragma unroll
      for (int s2 = 0; s2 < kStages; ++s2)
        if (s2 == s) last_issued[s2] = t;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(n * C::row_bytes));
      __syncwarp();
      unsigned char* st = data + s * C::stage_bytes;
      if (!p.paged) {
        const size_t base = ((size_t)b * p.Hkv + kvh) * (size_t)p.max_len + tr0;
        if (lane == 0)
          bulk_g2s(st, reinterpret_cast<const ET*>(p.k) + base * C::DN, (uint32_t)(n * C::DN * C::ES), &full[s], pol);
        if (DROT > 0 && lane == 1)
          bulk_g2s(st + C::kN, reinterpret_cast<const ET*>(p.k_rot) + ((size_t)b * p.max_len + tr0) * DROT,
                   (uint32_t)(n * DROT * C::ES), &full[s], pol);
        if (lane == 2)
          bulk_g2s(st + C::kN + C::kR, reinterpret_cast<const ET*>(p.v) + base * DV, (uint32_t)(n * DV * C::ES),
                   &full[s], pol);
      } else {
        const int blk0 = tr0 / p.bs, blk1 = (tr0 + n - 1) / p.bs;
        for (int bi = blk0 + lane; bi <= blk1; bi += 32) {
          const int ra = max(tr0, bi * p.bs), rz = min(tr0 + n, (bi + 1) * p.bs);
          const int e = p.tables[(size_t)b * p.mbps + bi];
          const size_t src_row = ((size_t)e * p.Hkv + kvh) * p.bs + (ra - bi * p.bs);
          bulk_g2s(st + (ra - tr0) * C::DN * C::ES, reinterpret_cast<const ET*>(p.k) + src_row * DK,
                   (uint32_t)((rz - ra) * DK * C::ES), &full[s], pol);
          bulk_g2s(st + C::kN + C::kR + (ra - tr0) * DV * C::ES, reinterpret_cast<const ET*>(p.v) + src_row * DV,
                   (uint32_t)((rz - ra) * DV * C::ES), &full[s], pol);
        }
      }
    }
    // Never leave with a copy in flight: wait (bounded) for the last tile
    // issued into each stage. On the normal path these have all completed.
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < kStages; ++s)
        if (last_issued[s] >= 0 && !mbar_wait(&full[s], (last_issued[s] / kStages) & 1)) {
          *abort_flag = 1;
          raise_error(p.err, kErrTimeout);
        }
    }
  } else {
    // ================= compute warps =================
    float2 q2[NV][H2K];
    int lim_own = 0;
#pragma unroll
    for (int vh = 0; vh < NV; ++vh) {
      const int iq = i0 + vh / p.GH;
      const int h = kvh * p.G + hc * p.GH + vh % p.GH;
      const bool active = iq <= i_last;
      if (vh == own) lim_own = active ? kv_len - p.seq_q + iq + 1 : 0;
      const ET* qrow = reinterpret_cast<const ET*>(p.q) + (((size_t)b * p.seq_q + (active ? iq : i0)) * p.H + h) * DK;
      const float qs = active ? p.qscale : 0.f;
#pragma unroll
      for (int qk = 0; qk < C::QK; ++qk) {
        float2 f[CH / 2];
        chunk_to_f2<ET>(__ldg(reinterpret_cast<const uint4*>(qrow + (li + L * qk) * CH)), f);
#pragma unroll
        for (int e = 0; e < CH / 2; ++e) q2[vh][qk * (CH / 2) + e] = make_float2(f[e].x * qs, f[e].y * qs);
      }
    }
    const int gbase = rgw * L;  // first lane of this row group
    const int rg = warp * C::RGW + rgw;

    for (int t = 0; t < ntiles; ++t) {
      const int s = t % kStages;
      if (!warp_wait(&full[s], (t / kStages) & 1, abort_flag, p.err)) break;
      const int tr0 = r0 + t * T;
      const int n = min(T, r1 - tr0);
      const unsigned char* st = data + s * C::stage_bytes;
      const ET* sKn = reinterpret_cast<const ET*>(st);
      const ET* sKr = reinterpret_cast<const ET*>(st + C::kN);
      const ET* sV = reinterpret_cast<const ET*>(st + C::kN + C::kR);
      // the two rows of this row group in the tile
      const int ra = rg, rb2 = rg + C::NRG;
      const bool va = ra < n, vb = rb2 < n;
      const int rra = va ? ra : 0, rrb = vb ? rb2 : 0;
      if (__any_sync(0xffffffffu, va)) {  // warp-uniform: some row of this warp is in the tile
        // ---- scores: NV partial dot products per row
        float2 acc_a[NV], acc_b[NV];  // paired partial sums, folded once per row
#pragma unroll
        for (int vh = 0; vh < NV; ++vh) acc_a[vh] = acc_b[vh] = make_float2(0.f, 0.f);
#pragma unroll
        for (int qk = 0; qk < C::QK; ++qk) {
          const int c = li + L * qk;
          const ET* srcA = (DROT == 0 || qk < C::NCH / L) ? sKn + rra * C::DN + c * CH
                                                           : sKr + rra * DROT + (c - C::NCH) * CH;
          const ET* srcB = (DROT == 0 || qk < C::NCH / L) ? sKn + rrb * C::DN + c * CH
                                                           : sKr + rrb * DROT + (c - C::NCH) * CH;
          float2 ka[CH / 2], kb[CH / 2];
          chunk_to_f2<ET>(*reinterpret_cast<const uint4*>(srcA), ka);
          chunk_to_f2<ET>(*reinterpret_cast<const uint4*>(srcB), kb);
#pragma unroll
          for (int vh = 0; vh < NV; ++vh)
#pragma unroll
            for (int e = 0; e < CH / 2; ++e) {
              acc_a[vh] = __ffma2_rn(q2[vh][qk * (CH / 2) + e], ka[e], acc_a[vh]);
              acc_b[vh] = __ffma2_rn(q2[vh][qk * (CH / 2) + e], kb[e], acc_b[vh]);
            }
        }
        float pa[NV], pb[NV];
#pragma unroll
        for (int vh = 0; vh < NV; ++vh) {
          pa[vh] = acc_a[vh].x + acc_a[vh].y;
          pb[vh] = acc_b[vh].x + acc_b[vh].y;
        }
        const float sa = reduce_own<NV, L>(pa, li);
        const float sb = reduce_own<NV, L>(pb, li);
        // ---- online softmax of the owned head over the two rows
        const bool visa = va && tr0 + ra < lim_own;
        const bool visb = vb && tr0 + rb2 < lim_own;
        const float mx = fmaxf(visa ? sa : -INFINITY, visb ? sb : -INFINITY);
        const bool grow = mx > m_ref + kRescaleLog2;
        float f = 1.f;
        if (grow) {
          f = ex2(m_ref - mx);  // 0 while m_ref = -inf
          l_sum *= f;
          m_ref = mx;
        }
        const float ea = visa ? ex2(sa - m_ref) : 0.f;
        const float eb = visb ? ex2(sb - m_ref) : 0.f;
        l_sum += ea + eb;
        if (__any_sync(0xffffffffu, grow)) {  // rare: move every head's accumulators to its new max
#pragma unroll
          for (int vh = 0; vh < NV; ++vh) {
            const float fh = NV == 1 ? f : __shfl_sync(0xffffffffu, f, gbase + owner_lane<NV, L>(vh));
#pragma unroll
            for (int e = 0; e < H2V; ++e) o2[vh][e] = make_float2(o2[vh][e].x * fh, o2[vh][e].y * fh);
          }
        }
        // ---- probabilities to every lane of the group, then P.V
        float2 pp[NV];
#pragma unroll
        for (int vh = 0; vh < NV; ++vh) {
          const float xa = NV == 1 ? ea : __shfl_sync(0xffffffffu, ea, gbase + owner_lane<NV, L>(vh));
          const float xb = NV == 1 ? eb : __shfl_sync(0xffffffffu, eb, gbase + owner_lane<NV, L>(vh));
          pp[vh] = make_float2(xa, xb);
        }
#pragma unroll
        for (int qv = 0; qv < C::QV; ++qv) {
          float2 fa[CH / 2], fb[CH / 2];
          chunk_to_f2<ET>(*reinterpret_cast<const uint4*>(sV + rra * DV + (li + L * qv) * CH), fa);
          chunk_to_f2<ET>(*reinterpret_cast<const uint4*>(sV + rrb * DV + (li + L * qv) * CH), fb);
#pragma unroll
          for (int vh = 0; vh < NV; ++vh) {
            const float2 wa = make_float2(pp[vh].x, pp[vh].x), wb = make_float2(pp[vh].y, pp[vh].y);
#pragma unroll
            for (int e = 0; e < CH / 2; ++e) {
              float2& acc = o2[vh][qv * (CH / 2) + e];
              acc = __ffma2_rn(wa, fa[e], acc);
              acc = __ffma2_rn(wb, fb[e], acc);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  // Every copy has landed and every compute warp is done with the ring.
  __syncthreads();

  // ---- merge the row groups (fixed order) through shared memory
  float* mm = reinterpret_cast<float*>(data);  // [NRG][NV]
  float* ml = mm + C::NRG * NV;                // [NRG][NV]
  float* mo = ml + C::NRG * NV;                // [NRG][NV][DV]
  if (warp < kRowsWarps) {
    const int rg = warp * C::RGW + rgw;
    if (li == owner_lane<NV, L>(own)) {
      mm[rg * NV + own] = m_ref;
      ml[rg * NV + own] = l_sum;
    }
#pragma unroll
    for (int vh = 0; vh < NV; ++vh)
#pragma unroll
      for (int qv = 0; qv < C::QV; ++qv)
#pragma unroll
        for (int e = 0; e < CH / 2; e += 2)
          *reinterpret_cast<float4*>(&mo[(rg * NV + vh) * DV + (li + L * qv) * CH + 2 * e]) =
              make_float4(o2[vh][qv * (CH / 2) + e].x, o2[vh][qv * (CH / 2) + e].y,
                          o2[vh][qv * (CH / 2) + e + 1].x, o2[vh][qv * (CH / 2) + e + 1].y);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < NV * DV; idx += blockDim.x) {
    const int vh = idx / DV, d = idx % DV;
    const int iq = i0 + vh / p.GH;
    if (iq > i_last) continue;
    const int h = kvh * p.G + hc * p.GH + vh % p.GH;
    float M = -INFINITY;
    for (int g = 0; g < C::NRG; ++g) M = fmaxf(M, mm[g * NV + vh]);
    float ls = 0.f, os = 0.f;
    if (M != -INFINITY) {
      for (int g = 0; g < C::NRG; ++g) {
        const float mg = mm[g * NV + vh];
        const float w = (mg == -INFINITY) ? 0.f : ex2(mg - M);
        ls = fmaf(w, ml[g * NV + vh], ls);
        os = fmaf(w, mo[(g * NV + vh) * DV + d], os);
      }
    }
    const size_t row = ((size_t)b * p.seq_q + iq) * p.H + h;
    if (nsplit == 1) {
      reinterpret_cast<ET*>(p.out)[row * DV + d] = Elem<ET>::from_f32(ls > 0.f ? os / ls : 0.f);
    } else {
      float* P = p.partial + (row * p.max_splits + split) * (DV + 2);
      if (d == 0) {
        P[0] = M;
        P[1] = ls;
      }
      P[2 + d] = os;
    }
  }
}

// Host launcher of one instantiation.
template <typename ET, int DK, int DV, int DROT, int NV>
cudaError_t launch_rows_inst(const RowsParams& p, cudaStream_t st) {
  using C = RowsCfg<ET, DK, DV, DROT, NV>;
  auto kern = attn_rows_kernel<ET, DK, DV, DROT, NV>;
  int dev = 0;
  cudaGetDevice(&dev);
  static unsigned long long attr_done = 0;  // one bit per device
  if (dev < 64 && !(attr_done >> dev & 1ull)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::smem_bytes);
    if (e != cudaSuccess) return e;
    attr_done |= 1ull << dev;
  }
  const long long items = (long long)p.B * p.Hkv * p.n_hchunks * p.n_rblocks;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL || p.max_splits > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)items, (unsigned)p.max_splits);
  kern<<<grid, kRowsThreads, C::smem_bytes, st>>>(p);
  return cudaGetLastError();
}

}  // namespace gqa
