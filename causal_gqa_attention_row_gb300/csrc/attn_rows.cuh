// attn_rows.cuh -- SIMT split-K attention of query rows against a KV cache.
//
// The operation (kopitiam-runtime src/attention.rs, `attention_forward`,
// `causal_mask`, `repeat_kv_heads`): query head h reads KV head h / G; query row
// i at position offset + i sees keys 0..=offset + i; softmax over the visible
// keys of scale * q.k, then the weighted sum of V.
//
// Work units: (sequence b, KV head kvh, a chunk of GH of that KV head's G
// query heads, a block of QR query rows, a split of the key range). A unit's
// GH*QR = NV "virtual heads" (query row, query head) all read the SAME K/V
// rows, so each K/V row crosses HBM once per KV head however large the group
// (frink-models src/decoder/attn_block.rs and kopitiam's module doc: every
// query head of a group genuinely shares its KV head).
//
// Scheduling: the kernel is persistent, one CTA per resident slot. With a
// split-K workspace, a one-CTA plan kernel first lists the units that have keys
// (every full split, then every item's final partial split) and the CTAs take
// units from that list one at a time through an atomic ticket, so the work
// balances to within one unit whatever the length mix. Without one (a single
// split per item) CTA c takes items c, c + grid, ... The producer warp alone
// fetches units; each tile it passes through the ring carries the unit's
// coordinates, so the compute warps simply follow the ring, and the copies of
// the next unit stream in while they merge the current one. A unit's first tile
// also brings its query rows into shared memory.
//
// Data path: one producer warp streams K/V tiles of T rows into an NS-deep
// shared-memory ring with 1-D bulk copies (cp.async.bulk, the TMA engine)
// completing on mbarriers. Contiguous caches need one copy per tile and
// operand; paged caches one per block segment, the block-table gather done by
// the copy engine (frink-models src/decoder/attn_block.rs, `push_and_attend_row`,
// paged arm). Four compute warps consume the ring. A unit whose block-table
// entries are out of range is caught by the producer before any of its copies;
// the producer then writes the unit's empty result itself.
//
// Compute mapping: a "row group" of L lanes owns one key row at a time; lane li
// works on the 16-byte chunks li, li+L, li+2L, ... of each row. It keeps its
// chunks of the output accumulators of every virtual head in registers, as
// float2 pairs for the paired FFMA2 instruction, and reads the matching chunks of
// q (fp32, pre-scaled by scale*log2 e) from its warp's copy in shared memory (the
// warp's row groups read the same addresses: 4-way broadcasts). Keeping q out of
// the registers lets three CTAs share an SM. A row's NV scores are L-lane
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
// unchanged. At the end of a unit the row groups of each warp are merged in
// registers (xor butterflies), then the warps through a shared-memory area of
// their own (not the ring), always in the same order (log-sum-exp); the result
// is written as the output (one split) or as a partial (m, l, o) that the
// combine kernel merges, again in a fixed order.
//
// The arms of the attention row (a template flag, so that plain calls run code
// without them): the owner lane applies a logit softcap and then an ALiBi bias
// to its head's score; a sliding window is a lower bound on the visible keys
// and on the tiles a unit streams; a sink logit joins the softmax denominator
// in the final merge (single split) or in the combine kernel.
//
// Determinism: split boundaries are multiples of kSplitRows, tiles multiples of
// T rows from the split start, and the row -> row-group assignment a function of
// the key index only. The arithmetic on a key row therefore does not depend on
// where the row lives (contiguous or paged), on the block table, on the other
// sequences of the batch or on which CTA takes the unit: paged and contiguous
// results are bit-identical, and so are repeated calls.
#pragma once

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace gqa {

constexpr int kRowsWarps = 4;  // compute warps
constexpr int kRowsThreads = (kRowsWarps + 1) * 32;
constexpr int kMaxStages = 4;
constexpr int kSmemBudget = 74 * 1024;  // shared memory per CTA (three CTAs per SM)
constexpr int kSmemPerSM = 228 * 1024;  // shared memory of one SM
constexpr int kSmemPerCTAReserved = 1024;
constexpr float kRescaleLog2 = 8.0f;

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int clog2(int x) { return x <= 1 ? 0 : 1 + clog2(x / 2); }

// Shared-memory header of the attention kernel.
struct RowsHeader {
  uint64_t full[kMaxStages];   // a tile has landed in the stage
  uint64_t empty[kMaxStages];  // the compute warps are done with the stage
  uint64_t merge[2];           // merge area: written / read by every compute warp
  int abort_flag;
  int pad_;
  // Per stage, the tile it holds: {item (-1: no more work), split, first key row,
  // rows | first tile of its unit << 16 | last tile << 17}.
  int4 tile[kMaxStages];
};

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
  static constexpr int kQ = NV * DK * ES;  // the unit's query rows, carried by its first tile
  static constexpr int stage_bytes = kN + kR + kV + kQ;
  static constexpr int row_bytes = (DN + DROT + DV) * ES;
  static constexpr int kHeader = 256;  // RowsHeader
  static constexpr int merge_bytes = kRowsWarps * NV * (DV + 2) * 4;  // one (m, l, o) per warp and head
  static constexpr int qbuf_bytes = kRowsWarps * NV * DK * 4;         // each warp's fp32 queries
  static constexpr int NS = cmax(
      2, cmin(kMaxStages, (kSmemBudget - kHeader - merge_bytes - qbuf_bytes) / stage_bytes));  // ring depth
  static constexpr int ring_bytes = NS * stage_bytes;
  static constexpr int smem_bytes = kHeader + ring_bytes + qbuf_bytes + merge_bytes;
  // CTAs per SM the register budget targets: three where shared memory allows.
  static constexpr int MIN_CTAS = cmax(1, cmin(3, kSmemPerSM / (smem_bytes + kSmemPerCTAReserved)));
  static_assert(DK % CH == 0 && DV % CH == 0 && DN % CH == 0, "head widths must be whole 16-byte chunks");
  static_assert(KCH % L == 0 && VCH % L == 0 && NCH % L == 0, "chunks must split evenly over a row group");
  static_assert(32 % L == 0, "row groups must tile a warp");
  static_assert(NV <= L, "a row group needs at least one lane per virtual head");
  static_assert(kSplitRows % T == 0, "split boundaries must fall on tile boundaries");
  static_assert(sizeof(RowsHeader) <= kHeader, "the header must fit its reserved space");
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

// 1/x on the special-function unit (the PTX rcp.approx instruction; 1/inf = 0).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// cap * tanh(s / cap) for a score s and cap in the log2 domain, with k = 2 log2(e) / cap:
// tanh(t) = 1 - 2 / (e^(2t) + 1), from 2^x and 1/x (absolute error near 1e-6 in
// tanh over the whole range; e^(2t) -> inf gives cap, -> 0 gives -cap).
__device__ __forceinline__ float softcap_log2(float s, float cap, float k) {
  return fmaf(-2.f * cap, rcp_approx(ex2(s * k) + 1.f), cap);
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

// One work unit: split `split` of item `item` (sequence, KV head, head chunk,
// query-row block).
struct Unit {
  int b, kvh, hc, split;
  int kv_len, i0, i_last;
  int r0, r1;   // key rows [r0, r1) of this split
  int lo;       // first key the unit's first row sees (the window's lower end)
  int nsplit;   // splits of the item that hold a visible key
  bool len_ok;
};

__device__ __forceinline__ Unit decode_unit(const RowsParams& p, int item, int split) {
  Unit u;
  u.split = split;
  const int rb = item % p.n_rblocks;
  item /= p.n_rblocks;
  u.hc = item % p.n_hchunks;
  item /= p.n_hchunks;
  u.kvh = item % p.Hkv;
  u.b = item / p.Hkv;
  u.kv_len = p.kv_len ? __ldg(p.kv_len + u.b) : (p.offsets ? __ldg(p.offsets + u.b) : 0) + p.seq_q;
  u.i0 = rb * p.QR;
  u.i_last = min(u.i0 + p.QR, p.seq_q) - 1;
  u.len_ok = u.kv_len >= p.seq_q && u.kv_len >= 1 && u.kv_len <= p.capacity;
  const int kv_hi = u.len_ok ? u.kv_len - p.seq_q + u.i_last + 1 : 0;  // keys the last row sees
  u.lo = u.len_ok ? first_visible_key(u.kv_len - p.seq_q + u.i0, p.window) : 0;
  u.nsplit = (kv_hi + p.split_rows - 1) / p.split_rows - u.lo / p.split_rows;
  u.r0 = split * p.split_rows;
  u.r1 = min(u.r0 + p.split_rows, kv_hi);
  return u;
}

// Output row of virtual head vh of a unit (query row, query head).
__device__ __forceinline__ size_t unit_out_row(const RowsParams& p, const Unit& u, int vh) {
  const int iq = u.i0 + vh / p.GH;
  const int h = u.kvh * p.G + u.hc * p.GH + vh % p.GH;
  return ((size_t)u.b * p.seq_q + iq) * p.H + h;
}

// Bounded barrier of the compute warps on an mbarrier that counts one arrival
// per warp. A warp that has given up never arrives, so the others give up too
// (after the bounded wait) instead of hanging.
__device__ __forceinline__ bool compute_sync(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned* err) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  return warp_wait(bar, parity, abort_flag, err);
}

// ARMS: the window / softcap / sink / ALiBi code is compiled in (a plain call
// runs the instantiation without it, at the plain kernel's register count).
template <typename ET, int DK, int DV, int DROT, int NV, bool ARMS>
__global__ void __launch_bounds__(kRowsThreads, RowsCfg<ET, DK, DV, DROT, NV>::MIN_CTAS)
    attn_rows_kernel(const RowsParams p) {
  using C = RowsCfg<ET, DK, DV, DROT, NV>;
  constexpr int CH = C::CH, L = C::L, T = C::T, kStages = C::NS;
  constexpr int H2K = C::EK / 2, H2V = C::EV / 2;  // float2 pairs per lane
  extern __shared__ __align__(1024) unsigned char smem[];
  RowsHeader* hdr = reinterpret_cast<RowsHeader*>(smem);
  volatile int* abort_flag = &hdr->abort_flag;
  unsigned char* data = smem + C::kHeader;
  float* qbuf = reinterpret_cast<float*>(smem + C::kHeader + C::ring_bytes);  // [warp][NV][DK]
  float* mm = qbuf + kRowsWarps * NV * DK;                                    // merge area: m [warp][NV]
  float* ml = mm + kRowsWarps * NV;                                           // l [warp][NV]
  float* mo = ml + kRowsWarps * NV;                                           // o [warp][NV][DV]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&hdr->full[s], 1);
      mbar_init(&hdr->empty[s], kRowsWarps);
    }
    mbar_init(&hdr->merge[0], kRowsWarps);
    mbar_init(&hdr->merge[1], kRowsWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Launched as a programmatic dependent of the kernel before it in the stream
  // (the unit plan, or the append): the set-up above may overlap it; nothing
  // below reads global memory before it has completed.
  grid_dep_wait();
  __syncthreads();

  if (warp == kRowsWarps) {
    // ================= producer warp =================
    const uint64_t pol = l2_policy_evict_first();
    const int n_items = p.B * p.Hkv * p.n_hchunks * p.n_rblocks;
    const int n_units = p.sched ? __ldcg(p.sched + 1) : n_items;
    int last_issued[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) last_issued[s] = -1;
    int gt = 0;  // tiles through the ring so far, across units
    int next_static = blockIdx.x;
    bool stop = false;
    while (!stop) {
      // ---- the next unit
      int item, split;
      if (p.sched) {
        int k = 0;
        if (lane == 0) k = atomicAdd(p.sched, 1);
        k = __shfl_sync(0xffffffffu, k, 0);
        if (k >= n_units) break;
        const int2 uu = __ldcg(p.units + k);
        item = uu.x;
        split = uu.y;
      } else {
        if (next_static >= n_items) break;
        item = next_static;
        split = 0;
        next_static += gridDim.x;
      }
      const Unit u = decode_unit(p, item, split);
      if (!u.len_ok) {
        // Length out of range: record it, write zeros, touch no K/V.
        if (lane == 0 && split == 0 && item % (p.Hkv * p.n_hchunks * p.n_rblocks) == 0)
          raise_error(p.err, kErrBounds);
        for (int idx = lane; idx < NV * DV; idx += 32) {
          const int vh = idx / DV;
          if (u.i0 + vh / p.GH >= p.seq_q) continue;
          reinterpret_cast<ET*>(p.out)[unit_out_row(p, u, vh) * DV + idx % DV] = Elem<ET>::from_f32(0.f);
        }
        continue;
      }
      if (p.paged) {
        // every block-table entry of the unit is checked before any copy
        const int blk0 = max(u.r0, u.lo) / p.bs, blk1 = (u.r1 - 1) / p.bs;  // entries below the window go unread
        bool bad = false;
        for (int bi = blk0 + lane; bi <= blk1; bi += 32) {
          const int e = __ldg(p.tables + (size_t)u.b * p.mbps + bi);
          if (e < 0 || e >= p.num_blocks) bad = true;
        }
        if (__any_sync(0xffffffffu, bad)) {
          // An empty partial (m = -inf, l = 0) or zeros: no K/V row is read.
          if (lane == 0) raise_error(p.err, kErrBounds);
          for (int idx = lane; idx < NV * DV; idx += 32) {
            const int vh = idx / DV, d = idx % DV;
            if (u.i0 + vh / p.GH > u.i_last) continue;
            const size_t row = unit_out_row(p, u, vh);
            if (u.nsplit == 1) {
              reinterpret_cast<ET*>(p.out)[row * DV + d] = Elem<ET>::from_f32(0.f);
            } else {
              float* P = p.partial + (row * p.max_splits + u.split) * (DV + 2);
              if (d == 0) {
                P[0] = -INFINITY;
                P[1] = 0.f;
              }
              P[2 + d] = 0.f;
            }
          }
          continue;
        }
      }
      const int ntiles = (u.r1 - u.r0 + T - 1) / T;
      // tiles stay aligned to the split start (the arithmetic on a key row must
      // not depend on the window); the first one holds the window's lower end
      const int t0 = u.lo > u.r0 ? (u.lo - u.r0) / T : 0;
      const int qrows = u.i_last - u.i0 + 1;
      for (int t = t0; t < ntiles; ++t, ++gt) {
        const int s = gt % kStages;
        if (gt >= kStages) {
          bool ok = true;
          if (lane == 0) ok = (*abort_flag == 0) && mbar_wait(&hdr->empty[s], ((gt / kStages) - 1) & 1);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            if (lane == 0) {
              *abort_flag = 1;
              raise_error(p.err, kErrTimeout);
            }
            stop = true;
            break;
          }
        }
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) {
          stop = true;
          break;
        }
        if (p.debug_withhold && gt == 0) continue;  // test hook: this tile never arrives
#pragma unroll
        for (int s2 = 0; s2 < kStages; ++s2)
          if (s2 == s) last_issued[s2] = gt;
        const int tr0 = u.r0 + t * T;
        const int n = min(T, u.r1 - tr0);
        unsigned char* st = data + s * C::stage_bytes;
        if (lane == 0) {
          hdr->tile[s] = make_int4(item, split, tr0, n | (t == t0 ? 1 << 16 : 0) | (t == ntiles - 1 ? 1 << 17 : 0));
          const uint32_t qb = t == t0 ? (uint32_t)(qrows * p.GH * DK * C::ES) : 0u;
          mbar_arrive_expect_tx(&hdr->full[s], (uint32_t)(n * C::row_bytes) + qb);
        }
        __syncwarp();
        if (!p.paged) {
          const size_t base = ((size_t)u.b * p.Hkv + u.kvh) * (size_t)p.max_len + tr0;
          if (lane == 0)
            bulk_g2s(st, reinterpret_cast<const ET*>(p.k) + base * C::DN, (uint32_t)(n * C::DN * C::ES),
                     &hdr->full[s], pol);
          if (DROT > 0 && lane == 1)
            bulk_g2s(st + C::kN, reinterpret_cast<const ET*>(p.k_rot) + ((size_t)u.b * p.max_len + tr0) * DROT,
                     (uint32_t)(n * DROT * C::ES), &hdr->full[s], pol);
          if (lane == 2)
            bulk_g2s(st + C::kN + C::kR, reinterpret_cast<const ET*>(p.v) + base * DV, (uint32_t)(n * DV * C::ES),
                     &hdr->full[s], pol);
        } else {
          const int blk0 = tr0 / p.bs, blk1 = (tr0 + n - 1) / p.bs;
          for (int bi = blk0 + lane; bi <= blk1; bi += 32) {
            const int ra = max(tr0, bi * p.bs), rz = min(tr0 + n, (bi + 1) * p.bs);
            // A block wholly below the window may be gone from the table; its rows
            // (masked out) are filled from the block holding the window's first
            // key, whose entry was checked, so that they hold finite values.
            const int bsrc = (bi + 1) * p.bs <= u.lo ? u.lo / p.bs : bi;
            const int e = __ldg(p.tables + (size_t)u.b * p.mbps + bsrc);
            const size_t src_row = ((size_t)e * p.Hkv + u.kvh) * p.bs + (ra - bi * p.bs);
            bulk_g2s(st + (ra - tr0) * C::DN * C::ES, reinterpret_cast<const ET*>(p.k) + src_row * DK,
                     (uint32_t)((rz - ra) * DK * C::ES), &hdr->full[s], pol);
            bulk_g2s(st + C::kN + C::kR + (ra - tr0) * DV * C::ES, reinterpret_cast<const ET*>(p.v) + src_row * DV,
                     (uint32_t)((rz - ra) * DV * C::ES), &hdr->full[s], pol);
          }
        }
        if (t == t0 && lane < qrows) {
          // query row i0 + lane: the unit's GH heads of it, contiguous
          const ET* src = reinterpret_cast<const ET*>(p.q) +
                          (((size_t)u.b * p.seq_q + u.i0 + lane) * p.H + u.kvh * p.G + u.hc * p.GH) * DK;
          bulk_g2s(st + C::kN + C::kR + C::kV + lane * p.GH * DK * C::ES, src, (uint32_t)(p.GH * DK * C::ES),
                   &hdr->full[s], pol);
        }
      }
    }
    if (!stop) {
      // end of work: one more tile descriptor, carrying no data
      const int s = gt % kStages;
      bool ok = true;
      if (lane == 0) {
        if (gt >= kStages) ok = (*abort_flag == 0) && mbar_wait(&hdr->empty[s], ((gt / kStages) - 1) & 1);
        if (ok) {
          hdr->tile[s] = make_int4(-1, 0, 0, 0);
          mbar_arrive(&hdr->full[s]);
        } else {
          *abort_flag = 1;
          raise_error(p.err, kErrTimeout);
        }
      }
      // The marker completes a phase of its stage: the drain below must wait
      // on that phase, not on the one before it (a parity wait cannot tell a
      // phase from the one two later).
      ok = __shfl_sync(0xffffffffu, ok, 0);
#pragma unroll
      for (int s2 = 0; s2 < kStages; ++s2)
        if (ok && s2 == s) last_issued[s2] = gt;
    }
    // Never leave with a copy in flight: wait (bounded) for the last tile
    // issued into each stage. On the normal path these have all completed.
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < kStages; ++s)
        if (last_issued[s] >= 0 && !mbar_wait(&hdr->full[s], (last_issued[s] / kStages) & 1)) {
          *abort_flag = 1;
          raise_error(p.err, kErrTimeout);
        }
    }
    return;
  }

  // ================= compute warps =================
  const int rgw = lane / L, li = lane % L;
  const int own = owned_head<NV, L>(li);  // the virtual head whose softmax this lane runs
  const int gbase = rgw * L;              // first lane of this row group
  const int rg = warp * C::RGW + rgw;
  const int ctid = threadIdx.x;           // 0 .. 32*kRowsWarps-1

  // This warp's copy of the unit's queries, fp32 and pre-scaled by scale*log2 e;
  // the four row groups read it as 4-way broadcasts.
  float* qw = qbuf + warp * NV * DK;
  // output accumulators (all heads, this lane's chunks) and the owned head's state
  float2 o2[NV][H2V];
  float m_ref = -INFINITY, l_sum = 0.f;
  int lim_own = 0;    // keys < lim_own are causal for the owned head's row
  int lo_own = 0;     // ... and keys >= lo_own inside its window
  float slope2 = 0.f; // the owned head's ALiBi slope in the log2 domain
  const float cap_k = ARMS && p.softcap2 > 0.f ? 2.8853900817779268f / p.softcap2 : 0.f;  // 2 log2(e) / cap
  int merges = 0;
  for (int gt = 0;; ++gt) {
    const int s = gt % kStages;
    if (!warp_wait(&hdr->full[s], (gt / kStages) & 1, abort_flag, p.err)) break;
    const int4 dsc = hdr->tile[s];
    if (dsc.x < 0) break;  // no more work
    const int tr0 = dsc.z, n = dsc.w & 0xffff;
    const unsigned char* st = data + s * C::stage_bytes;
    if (dsc.w & (1 << 16)) {
      // first tile of a unit: fresh state, queries from the stage into qw
      const Unit u = decode_unit(p, dsc.x, dsc.y);
      const ET* sQ = reinterpret_cast<const ET*>(st + C::kN + C::kR + C::kV);
      for (int idx = lane; idx < NV * DK; idx += 32) {
        const bool active = u.i0 + (idx / DK) / p.GH <= u.i_last;
        qw[idx] = active ? Elem<ET>::to_f32(sQ[idx]) * p.qscale : 0.f;
      }
#pragma unroll
      for (int vh = 0; vh < NV; ++vh) {
#pragma unroll
        for (int e = 0; e < H2V; ++e) o2[vh][e] = make_float2(0.f, 0.f);
        const int iq = u.i0 + vh / p.GH;
        if (vh == own) {
          lim_own = iq <= u.i_last ? u.kv_len - p.seq_q + iq + 1 : 0;
          if (ARMS) {
            lo_own = first_visible_key(lim_own - 1, p.window);
            slope2 = p.alibi ? __ldg(p.alibi + u.kvh * p.G + u.hc * p.GH + vh % p.GH) * kLog2e : 0.f;
          }
        }
      }
      m_ref = -INFINITY;
      l_sum = 0.f;
      __syncwarp();
    }
    {
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
          for (int vh = 0; vh < NV; ++vh) {
            const float4* qp = reinterpret_cast<const float4*>(qw + vh * DK + c * CH);
#pragma unroll
            for (int j = 0; j < CH / 4; ++j) {
              const float4 qq = qp[j];
              acc_a[vh] = __ffma2_rn(make_float2(qq.x, qq.y), ka[2 * j], acc_a[vh]);
              acc_b[vh] = __ffma2_rn(make_float2(qq.x, qq.y), kb[2 * j], acc_b[vh]);
              acc_a[vh] = __ffma2_rn(make_float2(qq.z, qq.w), ka[2 * j + 1], acc_a[vh]);
              acc_b[vh] = __ffma2_rn(make_float2(qq.z, qq.w), kb[2 * j + 1], acc_b[vh]);
            }
          }
        }
        float pa[NV], pb[NV];
#pragma unroll
        for (int vh = 0; vh < NV; ++vh) {
          pa[vh] = acc_a[vh].x + acc_a[vh].y;
          pb[vh] = acc_b[vh].x + acc_b[vh].y;
        }
        float sa = reduce_own<NV, L>(pa, li);
        float sb = reduce_own<NV, L>(pb, li);
        // ---- the arms: softcap on the scaled score, then the ALiBi bias
        if (ARMS && p.softcap2 > 0.f) {
          sa = softcap_log2(sa, p.softcap2, cap_k);
          sb = softcap_log2(sb, p.softcap2, cap_k);
        }
        if (ARMS && p.alibi) {
          sa = fmaf(slope2, (float)(tr0 + ra - (lim_own - 1)), sa);
          sb = fmaf(slope2, (float)(tr0 + rb2 - (lim_own - 1)), sb);
        }
        // ---- online softmax of the owned head over the two rows
        const bool visa = va && tr0 + ra < lim_own && (!ARMS || tr0 + ra >= lo_own);
        const bool visb = vb && tr0 + rb2 < lim_own && (!ARMS || tr0 + rb2 >= lo_own);
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
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&hdr->empty[s]);
    if (!(dsc.w & (1 << 17))) continue;

    // ---- last tile of the unit: merge, in a fixed order. First the RGW row
    // groups of this warp, in registers: xor butterflies over the lane bits
    // above the row group, after which every lane holds the same sums.
    float Mw[NV], lw[NV];
#pragma unroll
    for (int vh = 0; vh < NV; ++vh) {
      const float mg = NV == 1 ? m_ref : __shfl_sync(0xffffffffu, m_ref, gbase + owner_lane<NV, L>(vh));
      const float lg = NV == 1 ? l_sum : __shfl_sync(0xffffffffu, l_sum, gbase + owner_lane<NV, L>(vh));
      float M = mg;
#pragma unroll
      for (int off = L; off < 32; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      const float w = (mg == -INFINITY) ? 0.f : ex2(mg - M);
      float lsum = w * lg;
#pragma unroll
      for (int off = L; off < 32; off <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      Mw[vh] = M;
      lw[vh] = lsum;
#pragma unroll
      for (int e = 0; e < H2V; ++e) {
        float ox = o2[vh][e].x * w, oy = o2[vh][e].y * w;
#pragma unroll
        for (int off = L; off < 32; off <<= 1) {
          ox += __shfl_xor_sync(0xffffffffu, ox, off);
          oy += __shfl_xor_sync(0xffffffffu, oy, off);
        }
        o2[vh][e] = make_float2(ox, oy);
      }
    }
    // Then the warps, through the merge area.
    const uint32_t par = merges & 1;
    ++merges;
    // every warp is done reading the previous unit's merge area
    if (!compute_sync(&hdr->merge[0], par, abort_flag, p.err)) break;
    if (rgw == 0) {
      if (li == 0) {
#pragma unroll
        for (int vh = 0; vh < NV; ++vh) {
          mm[warp * NV + vh] = Mw[vh];
          ml[warp * NV + vh] = lw[vh];
        }
      }
#pragma unroll
      for (int vh = 0; vh < NV; ++vh)
#pragma unroll
        for (int qv = 0; qv < C::QV; ++qv)
#pragma unroll
          for (int e = 0; e < CH / 2; e += 2)
            *reinterpret_cast<float4*>(&mo[(warp * NV + vh) * DV + (li + L * qv) * CH + 2 * e]) =
                make_float4(o2[vh][qv * (CH / 2) + e].x, o2[vh][qv * (CH / 2) + e].y,
                            o2[vh][qv * (CH / 2) + e + 1].x, o2[vh][qv * (CH / 2) + e + 1].y);
    }
    if (!compute_sync(&hdr->merge[1], par, abort_flag, p.err)) break;
    const Unit u = decode_unit(p, dsc.x, dsc.y);
    for (int idx = ctid; idx < NV * DV; idx += kRowsWarps * 32) {
      const int vh = idx / DV, d = idx % DV;
      if (u.i0 + vh / p.GH > u.i_last) continue;
      float M = -INFINITY;
      for (int g = 0; g < kRowsWarps; ++g) M = fmaxf(M, mm[g * NV + vh]);
      float ls = 0.f, os = 0.f;
      if (M != -INFINITY) {
        for (int g = 0; g < kRowsWarps; ++g) {
          const float mg = mm[g * NV + vh];
          const float wg = (mg == -INFINITY) ? 0.f : ex2(mg - M);
          ls = fmaf(wg, ml[g * NV + vh], ls);
          os = fmaf(wg, mo[(g * NV + vh) * DV + d], os);
        }
      }
      const size_t row = unit_out_row(p, u, vh);
      if (u.nsplit == 1) {
        float res = ls > 0.f ? os / ls : 0.f;
        if (ARMS && p.sinks) {  // the sink logit joins the denominator (once per row and head)
          const float z2 = __ldg(p.sinks + u.kvh * p.G + u.hc * p.GH + vh % p.GH) * kLog2e;
          const float Mx = fmaxf(M, z2);
          const float a = M == -INFINITY ? 0.f : ex2(M - Mx);
          const float den = fmaf(ls, a, ex2(z2 - Mx));
          res = den > 0.f ? os * a / den : 0.f;
        }
        reinterpret_cast<ET*>(p.out)[row * DV + d] = Elem<ET>::from_f32(res);
      } else {
        float* P = p.partial + (row * p.max_splits + u.split) * (DV + 2);
        if (d == 0) {
          P[0] = M;
          P[1] = ls;
        }
        P[2 + d] = os;
      }
    }
  }
}

// Host launcher of one instantiation: a persistent grid of one CTA per
// resident slot (SMs x CTAs per SM), capped at the number of units.
template <typename ET, int DK, int DV, int DROT, int NV, bool ARMS>
cudaError_t launch_rows_inst_arms(const RowsParams& p, cudaStream_t st) {
  using C = RowsCfg<ET, DK, DV, DROT, NV>;
  auto kern = attn_rows_kernel<ET, DK, DV, DROT, NV, ARMS>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::atomic<int> slots_cache[64];  // per device, 0 = not yet known
  int slots = dev < 64 ? slots_cache[dev].load(std::memory_order_acquire) : 0;
  if (slots == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::smem_bytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRowsThreads, C::smem_bytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1 || sms < 1) return cudaErrorInvalidConfiguration;
    slots = per_sm * sms;
    if (dev < 64) slots_cache[dev].store(slots, std::memory_order_release);
  }
  const long long items = (long long)p.B * p.Hkv * p.n_hchunks * p.n_rblocks;
  if (items <= 0 || p.max_splits <= 0) return cudaSuccess;
  const long long units = p.sched ? items * p.max_splits : items;  // an upper bound with a plan
  if (items * p.max_splits > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int grid = (int)(units < slots ? units : slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kRowsThreads);
  cfg.dynamicSmemBytes = C::smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename ET, int DK, int DV, int DROT, int NV>
cudaError_t launch_rows_inst(const RowsParams& p, cudaStream_t st) {
  const bool arms = p.window > 0 || p.softcap2 > 0.f || p.sinks || p.alibi;
  return arms ? launch_rows_inst_arms<ET, DK, DV, DROT, NV, true>(p, st)
              : launch_rows_inst_arms<ET, DK, DV, DROT, NV, false>(p, st);
}

}  // namespace gqa
