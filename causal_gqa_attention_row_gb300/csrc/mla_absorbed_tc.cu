// mla_absorbed_tc.cu -- MLA decode in the absorbed (latent) form on the tcgen05
// tensor cores (bf16; latent width d_c = 512, rope width d_r = 64).
//
// The operation (frink-models src/mla/mod.rs, `absorbed_attention` and the
// `MlaKvB::Split` form): query head h of sequence b, already absorbed into the
// latent space (q_abs[b, h], width d_c + d_r), attends to the cache rows
// j < seq_len[b] of its sequence with softmax(scale * q_abs . row_j); a row is
// (c_j, k_rot_j), its key the whole row and its value c_j, the first d_c
// columns. Every head reads the same row (MQA with a group of H), so a row read
// from memory serves 2 * H * (2 d_c + d_r) flops: at H = 128 this is a
// contraction, not a stream, and it runs on the tensor cores.
//
// One cluster of two CTAs = one (sequence, tile of 128 heads, split of p.chunk
// cache rows); CTA r of the pair owns value columns [r d_c / 2, (r + 1) d_c / 2)
// and the heads are the MMA's 128 rows. Each CTA keeps the Q_abs columns of its
// value half plus the rope columns (5 of the 9 64-column blocks) and loads the
// same columns of each 64-row cache tile R, so the score contraction is split
// between the pair:
//   S_r = Q_abs[:, cols_r] R[:, cols_r]^T   M = 128 heads, N = 64 rows, K = 256 + 32
// (the rope block's 64 columns: the first 32 to CTA 0, the last 32 to CTA 1).
// The partial scores go through distributed shared memory: each softmax warp
// writes its rows of S_r into a local send buffer and moves them with one bulk
// copy into the peer's receive buffer (completing on the peer's barrier), and
// both CTAs form S = S_0 + S_1
// (one fp32 addition, the same bits on both sides), so the pair runs identical
// softmax arithmetic and agrees on every row max and sum. Then
//   O_r += P R[:, value half r]             M = 128 heads, N = 256, K = 64 rows
// with P (bf16) in tensor memory over the S columns it came from. A cache row
// is read from memory once per pair (each CTA fetches its 5 blocks), and no
// score is computed twice.
//
// Per CTA: shared memory holds Q_abs's 5 blocks (80 KiB, for the CTA's whole
// life), a two-stage ring of cache tiles (2 x 40 KiB) and the receive and send
// buffers of the exchange (2 x 32 KiB); tensor memory holds O (256 columns) and
// two S buffers (2 x 64).
// Roles (192 threads):
//   warps 0-3  softmax: thread t owns head h0 + t (TMEM lane t); warp w trades
//              its 32 rows with warp w of the peer
//   warp 4     initialises the barriers; TMA producer of Q_abs (once) and of
//              the cache tiles (lane i issues the box of local block i)
//   warp 5     allocates TMEM; one thread issues the MMAs, S_t as soon as its
//              tile has landed and PV_t as soon as P_t is in TMEM
// Softmax: a lazily moved reference max (threshold 2^8 in p), p rounded to
// bf16 and the fp32 row sum taken over exactly those p. Rows of the last tile at
// or past seq_len weigh zero, and their value rows in shared memory are zeroed
// before the PV MMA reads them, so whatever the cache holds past seq_len
// (within its capacity) cannot reach the output. A sequence with one split
// writes O / l as bf16; otherwise each split writes (m, l, O) in fp32 (m in the
// log2 domain) and the split-combine kernel merges them.

#include <atomic>
#include "tc_ptx.cuh"
#include "tmap.h"

namespace gqa {
namespace {

constexpr int kHeads = 128;    // query heads per cluster: the MMA's M
constexpr int kKeys = 64;      // cache rows per tile: the S MMA's N
constexpr int kStages = 2;     // cache-tile ring
constexpr int kThreads = 192;  // four softmax warps, the producer, the MMA warp
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kWaitHintNs = 20;

template <int DC, int DR>
struct MlaCfg {
  static constexpr int kW = DC + DR;            // row width
  static constexpr int kDVH = DC / 2;           // value columns per CTA
  static constexpr int kCBV = kDVH / 64;        // ... in 64-column blocks
  static constexpr int kCBR = DR / 64;          // rope blocks (shared by the pair)
  static constexpr int kCBL = kCBV + kCBR;      // blocks a CTA holds of a row
  static constexpr int kQBlk = kHeads * 128;    // one block of Q_abs: 128 rows x 128 bytes
  static constexpr int kRBlk = kKeys * 128;     // one block of a cache tile: 64 rows x 128 bytes
  static constexpr int kTileQ = kCBL * kQBlk;
  static constexpr int kTileR = kCBL * kRBlk;
  static constexpr int kXBuf = kHeads * kKeys * 4;  // 128 rows x 64 fp32: the receive buffer, then the send buffer
  static constexpr int kOffQ = 0, kOffR = kTileQ, kOffX = kOffR + kStages * kTileR;
  static constexpr int kOffBar = kOffX + 2 * kXBuf;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + alignment slack
  // K steps (16 columns) of the score MMA per CTA: its value blocks, and half of the rope blocks
  static constexpr int kStepsV = kCBV * 4, kStepsR = kCBR * 2;
  // TMEM columns: O, then the two S buffers (P over the first half of each)
  static constexpr uint32_t kColO = 0, kColS = kDVH;
  static_assert(DC % 128 == 0 && DR % 64 == 0, "whole 64-column blocks per half");
  static_assert(kDVH % 16 == 0 && kDVH <= 256, "one PV MMA covers the half");
  static_assert(kColS + 2 * kKeys <= kTmemCols, "TMEM map");
  static_assert(kSmemBytes <= 232448, "over the 227 KiB a CTA may use");
};

struct MlaParams {
  int B, H, max_len, chunk, max_splits, n_htiles;  // max_len: rows a sequence can hold
  const int32_t* seq_lens;  // [B] rows visible, >= 1 and <= max_len
  // paged cache (tables != NULL): a pool [num_blocks, bs, d_c + d_r]; row j of
  // sequence b in block tables[b * mbps + j / bs], slot j % bs; bs divides 64
  const int32_t* tables;
  int mbps, bs, num_blocks;
  float* partial;           // [B * H, max_splits, d_c + 2] when max_splits > 1
  __nv_bfloat16* out;       // [B, H, d_c]
  float qscale;             // attention_scale * log2(e)
  unsigned* err;
  int debug_withhold;       // test hook: CTA 1 of each pair never loads its first cache tile
};

struct MlaBars {
  uint64_t q_full, r_full[kStages], r_empty[kStages];
  uint64_t s_full[2], p_full[2], o_done[2], mma_final;
  // per softmax warp (its 32 rows, 8 KiB of each buffer):
  // x_full: the peer's partial rows have landed in this CTA's receive buffer
  //         (this warp's expected bytes, completed by the peer's bulk copy);
  // x_free: the peer has read the rows this CTA copied into its receive buffer
  //         (so that copy, and the read of this CTA's send buffer, are done)
  uint64_t x_full[4], x_free[4];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(MlaBars) <= 256, "barrier block");

// ---- cluster helpers ---------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared-memory address, in the cluster window, of `p` (an address of this
// CTA's shared memory) in the shared memory of CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Bulk copy of `bytes` from this CTA's shared memory into a peer CTA's; when
// they have landed they count as transaction bytes on the peer's mbarrier `bar`.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "r"(smem_u32(src)), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void arrive_cluster(uint32_t bar_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr) : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Probe of a phase with cluster-scope acquire (the peer's writes into this CTA's
// shared memory are visible once it succeeds).
__device__ __forceinline__ bool test_parity_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitHintNs)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool aborted(MlaBars* bars) {
  return *reinterpret_cast<volatile int*>(&bars->abort_flag);
}

__device__ __forceinline__ void abort_all(MlaBars* bars, unsigned* err) {
  *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
  raise_error(err, kErrTimeout);
}

__device__ __forceinline__ bool wait_quick(uint64_t* bar, uint32_t parity) {
  return mbar_test_parity_nb(bar, parity) || mbar_wait_hint(bar, parity, kWaitHintNs);
}

// One thread: bounded wait, the CTA aborts on a timeout.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, MlaBars* bars, unsigned* err) {
  if (aborted(bars)) return false;
  if (wait_quick(bar, parity)) return true;
  abort_all(bars, err);
  return false;
}

// Whole warp: every lane agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, MlaBars* bars, unsigned* err) {
  bool ok = !aborted(bars) && wait_quick(bar, parity);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) abort_all(bars, err);
  return ok;
}

// Whole warp, cluster-scope acquire, bounded.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, MlaBars* bars, unsigned* err) {
  bool ok = !aborted(bars);
  if (ok && !test_parity_cluster(bar, parity)) {
    const long long t0 = clock64();
    while (!(ok = test_parity_cluster(bar, parity))) {
      if (clock64() - t0 > kWaitLimitCycles || aborted(bars)) break;
    }
  }
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) abort_all(bars, err);
  return ok;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t ex2_bf16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// a += low bf16 of w, b += high bf16 of w, in fp32.
__device__ __forceinline__ void add_bf16x2(float& a, float& b, uint32_t w) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(a), "+f"(b)
      : "r"(w));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Byte offset of 16-byte chunk c of row r in an exchange buffer (rows of 256
// bytes; the chunk index XOR r % 16 spreads a warp's rows over the banks).
__device__ __forceinline__ uint32_t xchg_off(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 15)) * 16)); }

template <int DC, int DR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_absorbed_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_r,
                           const MlaParams p) {
  using C = MlaCfg<DC, DR>;
  extern __shared__ unsigned char smem_raw[];
  // swizzle atoms sit on 1024-byte boundaries of the shared window
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  MlaBars* bars = reinterpret_cast<MlaBars*>(smem + C::kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // launched as a programmatic dependent: the lengths and the query may come
  // from the kernel before this one
  grid_dep_wait();
  // ---- work item: the pair of one (sequence, head tile, split) is one cluster
  const int half = (int)cluster_rank();
  const uint32_t peer = (uint32_t)(half ^ 1);
  int rest = (int)(blockIdx.x >> 1);
  const int split = rest % p.max_splits;
  rest /= p.max_splits;
  const int ht = rest % p.n_htiles;
  const int b = rest / p.n_htiles;
  const int h0 = ht * kHeads;
  const int len = __ldg(p.seq_lens + b);
  const bool len_ok = len >= 1 && len <= p.max_len;
  const int n_split = len_ok ? (len + p.chunk - 1) / p.chunk : 1;
  if (split >= n_split) return;  // no rows in this split: both CTAs leave before any set-up
  if (!len_ok) {                 // the heads' output is zero and the error word says why
    if (threadIdx.x == 0 && half == 0 && ht == 0) raise_error(p.err, kErrBounds);
    for (int idx = threadIdx.x; idx < kHeads * C::kDVH; idx += blockDim.x) {
      const int h = h0 + idx / C::kDVH;
      if (h < p.H) p.out[((size_t)b * p.H + h) * DC + half * C::kDVH + idx % C::kDVH] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const int k0 = split * p.chunk;
  const int k1 = min(len, k0 + p.chunk);
  const int n_t = (k1 - k0 + kKeys - 1) / kKeys;  // >= 1

  // the global column block held in local block i: the value half, then the rope blocks
  auto global_block = [&](int i) { return i < C::kCBV ? half * C::kCBV + i : DC / 64 + (i - C::kCBV); };

  if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_init(&bars->q_full, 1);
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&bars->r_full[s], 1);
        mbar_init(&bars->r_empty[s], 1);
      }
      for (int x = 0; x < 2; ++x) {
        mbar_init(&bars->s_full[x], 1);
        mbar_init(&bars->p_full[x], 4);  // one arrival per softmax warp
        mbar_init(&bars->o_done[x], 1);
      }
      for (int w = 0; w < 4; ++w) {
        mbar_init(&bars->x_full[w], 1);
        mbar_init(&bars->x_free[w], 1);
      }
      mbar_init(&bars->mma_final, 1);
      bars->abort_flag = 0;
      fence_barrier_init();
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_r);
      mbar_arrive_expect_tx(&bars->q_full, C::kTileQ);
    }
    __syncwarp();
    // Q_abs [B, H, W]: this CTA's blocks of rows h0..h0+127 (heads past H read as zeros)
    if (lane < C::kCBL)
      tc::tma_load_4d(smem + C::kOffQ + lane * C::kQBlk, &tm_q, global_block(lane) * 64, h0, b, 0, &bars->q_full);
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  cluster_sync();  // both CTAs' barriers exist before either arrives at the other's
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kProducerWarp) {
    // ================= TMA producer of the cache tiles =================
    int issued_last[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) issued_last[s] = -1;
    // paged: a tile is `per` pool blocks; lane x < per * kCBL issues the box of
    // block x % per and column block x / per (each box a whole number of 8-row
    // swizzle atoms, so the boxes land where one box of the tile would put them)
    const int per = p.tables ? kKeys / p.bs : 1;
    const int nbox = per * C::kCBL;
    for (int t = 0; t < n_t; ++t) {
      const int st = t % kStages;
      int blk[2] = {0, 0};
      if (p.tables) {  // the tile's table entries, fetched before waiting for the stage
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int x = lane + 32 * u;
          if (x >= nbox) continue;
          const int ti = (k0 + t * kKeys) / p.bs + x % per;
          // a block past the sequence, or an entry out of range (flagged), loads
          // from past the end of the pool: the TMA engine fills it with zeros
          int e = p.num_blocks;
          if (ti < p.mbps && ti * p.bs < len) {
            e = __ldg(p.tables + (size_t)b * p.mbps + ti);
            if (e < 0 || e >= p.num_blocks) {
              raise_error(p.err, kErrBounds);
              e = p.num_blocks;
            }
          }
          blk[u] = e;
        }
      }
      if (p.debug_withhold && t == 0 && half == 1) continue;  // test hook: tile 0 is never requested
      if (t >= kStages) {  // the stage is free once PV_{t-2} is done
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(&bars->r_empty[st], ((t / kStages) - 1) & 1, bars, p.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&bars->r_full[st], C::kTileR);
      __syncwarp();
      unsigned char* dst = smem + C::kOffR + st * C::kTileR;
      if (!p.tables) {
        // rows k0 + 64t .. +63 of sequence b; rows past the cache's capacity read as zeros
        if (lane < C::kCBL)
          tc::tma_load_4d(dst + lane * C::kRBlk, &tm_r, global_block(lane) * 64, k0 + t * kKeys, b, 0,
                          &bars->r_full[st]);
      } else {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int x = lane + 32 * u;
          if (x < nbox)
            tc::tma_load_4d(dst + (x / per) * C::kRBlk + (x % per) * p.bs * 128, &tm_r, global_block(x / per) * 64, 0,
                            blk[u], 0, &bars->r_full[st]);
        }
      }
      __syncwarp();
      issued_last[st] = t;
    }
    if (lane == 0) {  // never exit with a load in flight
      if (!mbar_wait(&bars->q_full, 0)) raise_error(p.err, kErrTimeout);
      for (int s = 0; s < kStages; ++s)
        if (issued_last[s] >= 0 && !mbar_wait(&bars->r_full[s], (issued_last[s] / kStages) & 1))
          raise_error(p.err, kErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA issuer =================
    if (lane == 0) {
      const uint32_t idS = tc::idesc_bf16_f32(kHeads, kKeys, false);
      const uint32_t idO = tc::idesc_bf16_f32(kHeads, C::kDVH, true);
      constexpr uint64_t kHi = tc::desc_sw128_hi(0, 1024);  // K-major: 8-row groups 1024 bytes apart
      const uint64_t dQ = kHi | tc::desc_addr(smem + C::kOffQ);
      const uint64_t dR0 = kHi | tc::desc_addr(smem + C::kOffR);
      // the value half as V: MN-major, 8-row groups 1024 bytes apart, its 64-column
      // blocks one cache-tile block (8 KiB) apart
      const uint64_t dV0 = tc::desc_sw128_hi(C::kRBlk, 1024) | tc::desc_addr(smem + C::kOffR);
      const uint32_t tO = tmem + C::kColO;
      auto issue_s = [&](int t) {  // S_{t%2} = this CTA's share of Q_abs R_t^T
        const int st = t % kStages;
        const uint32_t tS = tmem + C::kColS + (t & 1) * kKeys;
        tc::fence_after_sync();
        const uint64_t dR = dR0 + (uint64_t)((st * C::kTileR) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::kStepsV + C::kStepsR; ++kk) {
          // value blocks: all four steps of each; rope blocks: this CTA's two steps of each
          const int blk = kk < C::kStepsV ? kk / 4 : C::kCBV + (kk - C::kStepsV) / 2;
          const int step = kk < C::kStepsV ? kk % 4 : half * 2 + (kk - C::kStepsV) % 2;
          const uint32_t aq = blk * C::kQBlk + step * 32;
          const uint32_t ar = blk * C::kRBlk + step * 32;
          tc::mma_f16_ss(tS, dQ + (aq >> 4), dR + (ar >> 4), idS, kk > 0);
        }
        tc::mma_commit(&bars->s_full[t & 1]);
      };
      auto issue_pv = [&](int t) {  // O += P_t R_t[:, value half], 16 rows per instruction
        const int st = t % kStages;
        const uint32_t tP = tmem + C::kColS + (t & 1) * kKeys;
        tc::fence_after_sync();
        const uint64_t dV = dV0 + (uint64_t)((st * C::kTileR) >> 4);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc::mma_f16_ts(tO, tP + kk * 8, dV + kk * (2048 >> 4), idO, (t > 0 || kk > 0));
        tc::mma_commit(&bars->o_done[t & 1]);
        tc::mma_commit(&bars->r_empty[st]);  // the tile's stage is free once PV_t is done
      };
      bool ok = wait_or_abort(&bars->q_full, 0, bars, p.err);
      // S_t needs tile t in shared memory, which also means PV_{t-2} is done: S
      // buffer t % 2 (holding P_{t-2}) has been read. PV_t needs P_t. Each barrier
      // is probed for its phases in order and cannot run two phases ahead.
      int next_s = 0, next_pv = 0;
      long long idle_since = clock64();
      while (ok && next_pv < n_t) {
        bool progressed = false;
        if (next_s < n_t && mbar_test_parity_nb(&bars->r_full[next_s % kStages], (next_s / kStages) & 1)) {
          issue_s(next_s++);
          progressed = true;
        }
        if (next_pv < next_s && mbar_test_parity_nb(&bars->p_full[next_pv & 1], (next_pv >> 1) & 1)) {
          issue_pv(next_pv++);
          progressed = true;
        }
        if (progressed) {
          idle_since = clock64();
        } else if (aborted(bars)) {
          ok = false;
        } else if (clock64() - idle_since > kWaitLimitCycles) {
          abort_all(bars, p.err);
          ok = false;
        }
      }
      // every MMA issued above has completed before TMEM is released
      tc::mma_commit(&bars->mma_final);
      if (!mbar_wait(&bars->mma_final, 0)) raise_error(p.err, kErrTimeout);
    }
  } else {
    // ================= softmax: thread t owns head h0 + t =================
    const int r = warp * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    const float qs = p.qscale;
    const float th = kRescaleLog2 / qs;
    const float2 qs2 = make_float2(qs, qs);
    float m_ref = -INFINITY, l_run = 0.f;
    bool alive = true;
    int consumed = -1;    // the last tile whose partial rows from the peer this warp has read
    bool posted = false;  // the expected bytes of tile consumed + 1 are on x_full
    for (int t = 0; t < n_t; ++t) {
      const int x = t & 1;
      if (!warp_wait(&bars->s_full[x], (t >> 1) & 1, bars, p.err)) {
        alive = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t tS = tmem + lane_addr + C::kColS + x * kKeys;
      uint32_t sv[kKeys];
      tc::tmem_ld_32x32b_x32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tc::tmem_ld_32x32b_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tc::tmem_ld_wait();
      // ---- trade partial scores with the peer. This warp's rows go into the send
      // buffer (free once the peer has read the previous tile: that also means
      // the copy out of it is done), one bulk copy moves them into the peer's
      // receive buffer, and the peer's rows arrive in this CTA's.
      if (t >= 1 && !warp_wait_cluster(&bars->x_free[warp], (t - 1) & 1, bars, p.err)) {
        alive = false;
        break;
      }
      {
        unsigned char* recv = smem + C::kOffX;
        unsigned char* send = smem + C::kOffX + C::kXBuf;
        const uint32_t sbase = smem_u32(send);
#pragma unroll
        for (int c = 0; c < kKeys / 4; ++c)
          st_shared_v4(sbase + xchg_off(r, c), sv[4 * c], sv[4 * c + 1], sv[4 * c + 2], sv[4 * c + 3]);
        tc::fence_async_smem();  // the rows visible to the bulk copy
        __syncwarp();
        constexpr uint32_t kWarpBytes = 32 * kKeys * 4;
        if (lane == 0) {
          bulk_copy_to_peer(peer_addr(recv + warp * kWarpBytes, peer), send + warp * kWarpBytes, kWarpBytes,
                            peer_addr(&bars->x_full[warp], peer));
          mbar_arrive_expect_tx(&bars->x_full[warp], kWarpBytes);
        }
        posted = true;
        // S = S_0 + S_1
        if (!warp_wait_cluster(&bars->x_full[warp], t & 1, bars, p.err)) {
          alive = false;
          break;
        }
        const uint32_t lbase = smem_u32(recv);
#pragma unroll
        for (int c = 0; c < kKeys / 4; ++c) {
          const float4 o = ld_shared_v4(lbase + xchg_off(r, c));
          sv[4 * c] = __float_as_uint(__uint_as_float(sv[4 * c]) + o.x);
          sv[4 * c + 1] = __float_as_uint(__uint_as_float(sv[4 * c + 1]) + o.y);
          sv[4 * c + 2] = __float_as_uint(__uint_as_float(sv[4 * c + 2]) + o.z);
          sv[4 * c + 3] = __float_as_uint(__uint_as_float(sv[4 * c + 3]) + o.w);
        }
        consumed = t;
        posted = false;
        __syncwarp();
        if (lane == 0) arrive_cluster(peer_addr(&bars->x_free[warp], peer));
      }
      const int kt = k0 + t * kKeys;
      const int valid = min(kKeys, k1 - kt);  // rows of this tile the heads see
      if (valid < kKeys) {
#pragma unroll
        for (int e = 0; e < kKeys; ++e)
          if (e >= valid) sv[e] = __float_as_uint(-INFINITY);
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < kKeys; e += 2)
        mx4[(e >> 1) & 3] = fmax3(mx4[(e >> 1) & 3], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      if (t == 0) {
        m_ref = mx;  // the first tile has a visible row: mx is finite
      } else {
        const bool grow = mx > m_ref + th;
        if (__any_sync(0xffffffffu, grow)) {
          float f = 1.f;
          if (grow) {
            f = ex2f((m_ref - mx) * qs);
            m_ref = mx;
          }
          // O holds every PV issued so far, PV_{t-1} the last: rescale it once done
          if (!warp_wait(&bars->o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, bars, p.err)) {
            alive = false;
            break;
          }
          tc::fence_after_sync();
          uint32_t o[32];
#pragma unroll 1
          for (int c = 0; c < C::kDVH / 32; ++c) {
            tc::tmem_ld_32x32b_x32(tmem + lane_addr + C::kColO + c * 32, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tc::tmem_st_32x32b_x32(tmem + lane_addr + C::kColO + c * 32, o);
          }
          tc::tmem_st_wait();
          l_run *= f;
        }
      }
      // p = 2^(s*qs - m*qs) as bf16 pairs, and the fp32 sum of exactly these p
      const float mq = m_ref * qs;
      const float2 nmq2 = make_float2(-mq, -mq);
      uint32_t pv[kKeys / 2];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kKeys / 2; ++i) {
        const float2 xv = __ffma2_rn(make_float2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), qs2, nmq2);
        pv[i] = ex2_bf16x2(pack_bf16(xv.x, xv.y));
        add_bf16x2(ls[(i & 1) * 2], ls[(i & 1) * 2 + 1], pv[i]);
      }
      l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      if (valid < kKeys) {
        // value rows valid..63 of this CTA's half: zero them (S_t, their other
        // reader, is done) so that 0 * (whatever the cache holds) cannot be NaN
        unsigned char* base = smem + C::kOffR + (t % kStages) * C::kTileR;
        const int n_chunks = (kKeys - valid) * C::kCBV * 8;  // 16-byte chunks: 8 per row and block
        for (int i = r; i < n_chunks; i += kHeads) {
          const int row = valid + i / (C::kCBV * 8), blk = (i / 8) % C::kCBV, ch = i % 8;
          *reinterpret_cast<uint4*>(base + blk * C::kRBlk + row * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        tc::fence_async_smem();  // visible to the tensor cores' reads
      }
      // P_t over the first 32 columns of S buffer x (S_t has been read; PV_{t-2},
      // the last reader of P_{t-2} there, completed before S_t was issued)
      tc::tmem_st_32x32b_x16(tS, *reinterpret_cast<uint32_t(*)[16]>(&pv[0]));
      tc::tmem_st_32x32b_x16(tS + 16, *reinterpret_cast<uint32_t(*)[16]>(&pv[16]));
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[x]);
    }
    if (!alive && consumed + 1 < n_t) {
      // after a wait gave up: the peer may still be copying its rows of the next
      // tile into this CTA's receive buffer (at most that one copy: it needs this
      // warp's x_free for every earlier tile). Wait for it, bounded, so that no
      // copy lands after the CTA has exited.
      if (lane == 0 && !posted) mbar_arrive_expect_tx(&bars->x_full[warp], 32 * kKeys * 4);
      __syncwarp();
      const long long t0 = clock64();
      while (!test_parity_cluster(&bars->x_full[warp], (consumed + 1) & 1) && clock64() - t0 < kWaitLimitCycles) {
      }
    }
    // ---- the last PV (its commit covers every earlier MMA), then the output
    bool have_o = alive;
    if (have_o) {
      have_o = warp_wait(&bars->o_done[(n_t - 1) & 1], ((n_t - 1) >> 1) & 1, bars, p.err);
      tc::fence_after_sync();
    }
    const int h = h0 + r;
    const bool mine = h < p.H;
    if (n_split == 1) {
      const float inv = (have_o && l_run > 0.f) ? 1.f / l_run : 0.f;
      __nv_bfloat16* dst = p.out + ((size_t)b * p.H + (mine ? h : 0)) * DC + half * C::kDVH;
#pragma unroll 1
      for (int c = 0; c < C::kDVH / 32; ++c) {
        uint32_t o[32];
        tc::tmem_ld_32x32b_x32(tmem + lane_addr + C::kColO + c * 32, o);
        tc::tmem_ld_wait();
        if (mine) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              w[u] = pack_bf16(__uint_as_float(o[q4 * 8 + 2 * u]) * inv, __uint_as_float(o[q4 * 8 + 2 * u + 1]) * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + q4 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    } else {
      float* P = p.partial + (((size_t)b * p.H + (mine ? h : 0)) * p.max_splits + split) * (DC + 2);
      if (mine && half == 0) {
        P[0] = have_o ? m_ref * qs : -INFINITY;
        P[1] = have_o ? l_run : 0.f;
      }
      float* dst = P + 2 + half * C::kDVH;
#pragma unroll 1
      for (int c = 0; c < C::kDVH / 32; ++c) {
        uint32_t o[32];
        tc::tmem_ld_32x32b_x32(tmem + lane_addr + C::kColO + c * 32, o);
        tc::tmem_ld_wait();
        if (mine) {
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            *reinterpret_cast<float2*>(dst + c * 32 + e) = make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1]));
        }
      }
    }
  }

  grid_dep_launch();  // the split combine may start launching on freed SMs
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer's last accesses to this CTA's shared memory are done
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

// A bf16 tensor [d2, d1, w] (rows of w elements); box = 64 columns x box1 rows,
// 128-byte swizzle; rows and columns past the tensor read as zeros.
bool make_rows_map(CUtensorMap* m, const void* base, int w, uint64_t d1, uint64_t d2, uint32_t box1) {
  const uint64_t dims[4] = {(uint64_t)w, d1, d2, 1};
  const uint64_t strides[3] = {(uint64_t)w * 2, (uint64_t)w * 2 * d1, (uint64_t)w * 2 * d1 * d2};
  const uint32_t box[4] = {64, box1, 1, 1};
  return make_tmap_bf16(m, base, dims, strides, box);
}

}  // namespace

bool mla_absorbed_tc_supported(int bf16, int d_c, int d_r) { return bf16 == 1 && d_c == 512 && d_r == 64; }

bool mla_absorbed_paged_block_ok(int bs) { return bs > 0 && bs % 8 == 0 && kKeys % bs == 0; }

cudaError_t launch_mla_absorbed_tc(const void* q_abs, const void* latent, const int32_t* seq_lens, void* out_lat,
                                   float* partial, int B, int max_len, int H, int d_c, int d_r, int chunk,
                                   float qscale, unsigned* err, cudaStream_t st, const int32_t* tables, int mbps,
                                   int bs, int num_blocks, int debug_withhold) {
  using C = MlaCfg<512, 64>;
  if (!mla_absorbed_tc_supported(1, d_c, d_r) || chunk % kKeys != 0 || chunk <= 0 || !(qscale > 0.f))
    return cudaErrorNotSupported;
  if (tables && !mla_absorbed_paged_block_ok(bs)) return cudaErrorNotSupported;
  if (B == 0) return cudaSuccess;
  CUtensorMap tq, tr;
  // q_abs [B, H, 576]: box of 128 heads
  if (!make_rows_map(&tq, q_abs, C::kW, (uint64_t)H, (uint64_t)B, kHeads)) return cudaErrorInvalidValue;
  if (tables) {
    // pool [num_blocks, bs, 576]: box of one block
    if (!make_rows_map(&tr, latent, C::kW, (uint64_t)bs, (uint64_t)num_blocks, (uint32_t)bs)) return cudaErrorInvalidValue;
    max_len = mbps * bs;
  } else {
    // latent [B, max_len, 576]: box of one 64-row tile
    if (!make_rows_map(&tr, latent, C::kW, (uint64_t)max_len, (uint64_t)B, kKeys)) return cudaErrorInvalidValue;
  }
  MlaParams p;
  p.tables = tables;
  p.mbps = mbps;
  p.bs = bs;
  p.num_blocks = num_blocks;
  p.B = B;
  p.H = H;
  p.max_len = max_len;
  p.chunk = chunk;
  p.max_splits = (max_len + chunk - 1) / chunk;
  p.n_htiles = (H + kHeads - 1) / kHeads;
  p.seq_lens = seq_lens;
  p.partial = partial;
  p.out = static_cast<__nv_bfloat16*>(out_lat);
  p.qscale = qscale;
  p.err = err;
  p.debug_withhold = debug_withhold;
  int dev = 0;
  cudaGetDevice(&dev);
  static std::atomic<unsigned long long> attr_done{0};  // per device
  if (dev < 64 && !(attr_done.load(std::memory_order_acquire) >> dev & 1ull)) {
    const cudaError_t e =
        cudaFuncSetAttribute(mla_absorbed_tc_kernel<512, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(1ull << dev, std::memory_order_release);
  }
  const long long ctas = (long long)B * p.n_htiles * p.max_splits * 2;  // clusters of two
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);  // clusters of two (the kernel's __cluster_dims__)
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_absorbed_tc_kernel<512, 64>, tq, tr, p);
}

}  // namespace gqa
