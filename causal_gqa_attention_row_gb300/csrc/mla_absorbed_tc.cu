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
// cache rows); the heads are the MMA's 128 rows. The pair walks the split in
// tiles of 64 cache rows R_t and divides each tile two ways:
//   - the keys: CTA r scores rows 32r .. 32r + 31 of the tile against the whole
//     query row, S_r = Q_abs R_t[32r .. 32r + 31]^T (M = 128, N = 32, K = 576);
//   - the values: CTA r accumulates value columns [r d_c / 2, (r + 1) d_c / 2)
//     of all 64 rows, O_r += P R_t[:, value half r] (M = 128, N = 256, K = 64).
// So each CTA needs the other's P. The pair agrees on one reference max per
// head first: each CTA sends its tile row maxima (128 floats) to the other with
// asynchronous remote stores, both take the larger, and both then move the
// reference, rescale O and l, and form p = 2^(s*qs - m*qs) in bf16 the same
// way. Each CTA writes its 32 columns of P_t into the tile's shared-memory P
// and copies them, one bulk copy per softmax warp and 8-key column, into the
// same place of the peer's; the PV MMA reads P from there. Per tile a CTA sends
// 8.5 KiB to its peer (the bf16 P half and the maxima) instead of a fp32 score
// tile. Each CTA keeps the row sum of its own p; the two sums are added once,
// at the end.
//
// Per CTA: tensor memory holds O (256 columns), S (32) and the first 448 of the
// 576 Q_abs columns (224 columns, two bf16 per column: the score MMA's A
// operand). Shared memory holds the other two Q_abs column blocks (32 KiB) and
// two rings: R, four stages of the CTA's own 32 rows in full (36 KiB), and V,
// three stages of the peer's 32 rows' value half (16 KiB), needed only by the
// PV MMA. Once S_t is done the other half's value blocks of R stage t are
// dead, and P_t (16 KiB, no swizzle: each 8-key column of all 128 heads is
// 2 KiB, so a CTA's half is 4 contiguous pieces) is written over them. So P
// needs no buffer and no hand-over of its own: the peer copies its columns in
// only after it has this CTA's tile maxima, which are sent after S_t. The
// Q_abs blocks bound for TMEM arrive once, by TMA, in the part of the rings
// that the first tiles do not use (R stages 2 and 3, the V ring); each softmax
// thread moves its head's row from there into TMEM, and only then do tiles
// land there. The R ring is filled one tile ahead of the V ring.
// Roles (192 threads):
//   warps 0-3  softmax: thread t owns head h0 + t (TMEM lane t); warp w trades
//              maxima and P columns with warp w of the peer
//   warp 4     initialises the barriers; TMA producer of Q_abs (once) and of
//              the cache tiles
//   warp 5     allocates TMEM; issues the MMAs (one elected lane), S_t as soon
//              as its rows have landed and S_{t-1} has been read, PV_t once both
//              halves of P_t and the peer's rows are in place
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
constexpr int kKeys = 64;      // cache rows per tile of the pair
constexpr int kOwn = 32;       // ... of which each CTA scores 32: the S MMA's N
constexpr int kStagesR = 4;    // ring of this CTA's cache rows (and the P tiles)
constexpr int kStagesV = 3;    // ring of the peer rows' value halves
constexpr int kThreads = 192;  // four softmax warps, the producer, the MMA warp
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kWaitHintNs = 20;

template <int DC, int DR>
struct MlaCfg {
  static constexpr int kW = DC + DR;            // row width
  static constexpr int kNB = kW / 64;           // 64-column blocks of a row
  static constexpr int kDVH = DC / 2;           // value columns per CTA
  static constexpr int kCBV = kDVH / 64;        // ... in 64-column blocks
  static constexpr int kQS = 2;                 // Q_abs blocks in shared memory (the last two)
  static constexpr int kQT = kNB - kQS;         // ... and in tensor memory (the first seven)
  static constexpr int kQBlk = kHeads * 128;    // one block of Q_abs: 128 rows x 128 bytes
  static constexpr int kRBlk = kOwn * 128;      // one block of a CTA's cache rows: 32 rows x 128 bytes
  // a stage of the R ring: this CTA's 32 rows of a tile, every block; of the
  // V ring: the peer's 32 rows, this CTA's value blocks
  static constexpr int kStageR = kNB * kRBlk, kStageV = kCBV * kRBlk;
  // A tile's P (128 heads x 64 keys, bf16) goes into its R stage over the other
  // half's value blocks, which only the score MMA reads: kCBV blocks, 16 KiB.
  static constexpr int kPCol = kHeads * 16;  // one 8-key column of P: 2 KiB
  // shared memory: Q_abs's blocks, the two rings, maxima and row sums, barriers
  static constexpr int kOffQ = 0, kOffR = kOffQ + kQS * kQBlk, kOffV = kOffR + kStagesR * kStageR;
  static constexpr int kOffM = kOffV + kStagesV * kStageV;  // [2][128] maxima by tile parity, then [128] row sums
  static constexpr int kOffBar = kOffM + 3 * kHeads * 4;
  static constexpr int kSmemBytes = kOffBar + 384 + 1023;  // + alignment slack
  // At the start the kQT Q_abs blocks bound for TMEM land, by TMA, over R
  // stages 2 and 3 and the V ring; no cache tile is loaded there until every
  // softmax thread has moved its row into TMEM
  static constexpr int kOffStage = kOffR + 2 * kStageR;
  // TMEM columns: O, S, then Q_abs's first kQT blocks (32 columns each)
  static constexpr uint32_t kColO = 0, kColS = kDVH, kColQ = kColS + kOwn;
  static_assert(DC % 128 == 0 && DR % 64 == 0, "whole 64-column blocks per half");
  static_assert(kDVH % 16 == 0 && kDVH <= 256, "one PV MMA covers the half");
  static_assert(kColQ % 32 == 0 && kColQ + kQT * 32 <= kTmemCols, "TMEM map");
  static_assert(kOffR % 1024 == 0 && kStageR % 1024 == 0 && kOffV % 1024 == 0 && kStageV % 1024 == 0,
                "swizzle atoms on 1024-byte boundaries");
  static_assert(kCBV * kRBlk == kHeads * kKeys * 2, "P fills the other half's value blocks");
  static_assert(kSmemBytes <= 232448, "over the 227 KiB a CTA may use");
  static_assert(kOffStage % 1024 == 0 && kOffStage + kQT * kQBlk <= kOffM, "Q_abs staging inside the rings");
};

struct MlaParams {
  int B, H, max_len, chunk, max_splits, n_htiles;  // max_len: rows a sequence can hold
  const int32_t* seq_lens;  // [B] rows visible, >= 1 and <= max_len
  const __nv_bfloat16* q_abs;  // [B, H, d_c + d_r]
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
  // q_full: Q_abs's shared-memory blocks have landed and every softmax warp has
  // written its rows of the rest into TMEM (so their staging area is free);
  // q_stage: the rest has landed in the staging area
  uint64_t q_full, q_stage, r_full[kStagesR], v_full[kStagesV];
  // s_full / s_free: S_t is in TMEM / every softmax warp has read it;
  // p_full[x]: P_t is in place (this CTA's four warps and the peer's 8 KiB), t of parity x;
  // o_done[t % kStagesR]: PV_t is done, so O may be rescaled and R stage t % kStagesR
  // and V stage t % kStagesV refilled. One commit per PV: a second commit after
  // the same MMAs was seen to arrive up to ~1,600 cycles after the first.
  uint64_t s_full, s_free, p_full[2], o_done[kStagesR], mma_final;
  // per softmax warp w (its 32 heads):
  // m_full[w][x]: the peer's tile maxima for tile parity x have landed (128 bytes)
  // l_full[w]:    the peer's row sums have landed (once)
  uint64_t m_full[4][2], l_full[4];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(MlaBars) <= 384, "barrier block");

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

// Asynchronous 4-byte store into a peer CTA's shared memory, counted as
// transaction bytes on the peer's mbarrier `bar`.
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr), "r"(v),
               "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
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

template <int DC, int DR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_absorbed_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_r,
                           const __grid_constant__ CUtensorMap tm_v, const MlaParams p) {
  using C = MlaCfg<DC, DR>;
  extern __shared__ unsigned char smem_raw[];
  // swizzle atoms sit on 1024-byte boundaries of the shared window
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  MlaBars* bars = reinterpret_cast<MlaBars*>(smem + C::kOffBar);
  float* mbuf = reinterpret_cast<float*>(smem + C::kOffM);  // [2][kHeads]: the peer's tile maxima
  float* lbuf = mbuf + 2 * kHeads;                          // [kHeads]: the peer's row sums
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: the pair of one (sequence, head tile, split) is one cluster
  const int half = (int)cluster_rank();
  const uint32_t peer = (uint32_t)(half ^ 1);
  int rest = (int)(blockIdx.x >> 1);
  const int split = rest % p.max_splits;
  rest /= p.max_splits;
  const int ht = rest % p.n_htiles;
  const int b = rest / p.n_htiles;
  const int h0 = ht * kHeads;
  if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_init(&bars->q_full, 5);  // the producer's expected bytes + one arrival per softmax warp
      mbar_init(&bars->q_stage, 1);
      for (int s = 0; s < kStagesR; ++s) {
        mbar_init(&bars->r_full[s], 1);
      }
      for (int s = 0; s < kStagesV; ++s) {
        mbar_init(&bars->v_full[s], 1);
      }
      mbar_init(&bars->s_full, 1);
      mbar_init(&bars->s_free, 4);  // one arrival per softmax warp
      for (int x = 0; x < 2; ++x) mbar_init(&bars->p_full[x], 4);
      for (int s = 0; s < kStagesR; ++s) mbar_init(&bars->o_done[s], 1);
      mbar_init(&bars->mma_final, 1);
      for (int w = 0; w < 4; ++w) {
        for (int x = 0; x < 2; ++x) mbar_init(&bars->m_full[w][x], 1);
        mbar_init(&bars->l_full[w], 1);
      }
      bars->abort_flag = 0;
      fence_barrier_init();
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_r);
      tc::prefetch_tmap(&tm_v);
    }
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  cluster_sync();  // both CTAs' barriers exist before either arrives at the other's
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  // Launched as a programmatic dependent: the set-up above overlaps the end of
  // the kernel before this one, which may write the lengths, the query or the
  // cache; nothing global is read before it is complete.
  grid_dep_wait();
  const int len = __ldg(p.seq_lens + b);
  const bool len_ok = len >= 1 && len <= p.max_len;
  const int n_split = len_ok ? (len + p.chunk - 1) / p.chunk : 1;
  if (split >= n_split || !len_ok) {  // both CTAs of the pair (same sequence and split) leave here
    if (!len_ok) {                     // the heads' output is zero and the error word says why
      if (threadIdx.x == 0 && half == 0 && ht == 0) raise_error(p.err, kErrBounds);
      for (int idx = threadIdx.x; idx < kHeads * C::kDVH; idx += blockDim.x) {
        const int h = h0 + idx / C::kDVH;
        if (h < p.H) p.out[((size_t)b * p.H + h) * DC + half * C::kDVH + idx % C::kDVH] = __float2bfloat16_rn(0.f);
      }
    }
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);  // nothing was issued
    return;
  }
  const int k0 = split * p.chunk;
  const int k1 = min(len, k0 + p.chunk);
  const int n_t = (k1 - k0 + kKeys - 1) / kKeys;  // >= 1

  if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->q_full, C::kQS * C::kQBlk);
      mbar_arrive_expect_tx(&bars->q_stage, C::kQT * C::kQBlk);
    }
    __syncwarp();
    // Q_abs [B, H, W], rows h0..h0+127 (heads past H read as zeros): its last
    // kQS blocks where the score MMA reads them, the first kQT into the staging area
    if (lane < C::kQS)
      tc::tma_load_4d(smem + C::kOffQ + lane * C::kQBlk, &tm_q, (C::kQT + lane) * 64, h0, b, 0, &bars->q_full);
    else if (lane < C::kQS + C::kQT)
      tc::tma_load_4d(smem + C::kOffStage + (lane - C::kQS) * C::kQBlk, &tm_q, (lane - C::kQS) * 64, h0, b, 0,
                      &bars->q_stage);
  }

  if (warp == kProducerWarp) {
    // ================= TMA producer of the cache tiles =================
    // Tile t: this CTA's 32 rows (every block) into R stage t % kStagesR, and
    // the peer's 32 rows (this CTA's value blocks) into V stage t % kStagesV.
    // The latent is seen as [outer][row][column block][64], so a box of 32 rows
    // x several blocks lands block after block, as the MMAs read it: one box
    // per part (tm_r: all 9 blocks, tm_v: 4 value blocks). A paged pool of 8-
    // or 16-row blocks takes `per` boxes of `br` rows per column block instead
    // (tm_r then has a box of one block).
    int last_r[kStagesR], last_v[kStagesV];
#pragma unroll
    for (int s = 0; s < kStagesR; ++s) last_r[s] = -1;
#pragma unroll
    for (int s = 0; s < kStagesV; ++s) last_v[s] = -1;
    const int br = p.tables ? min(p.bs, kOwn) : kOwn;
    const int per = kOwn / br;
    const bool whole = per == 1;  // one box per part
    // The tensor-map coordinates (row or slot, sequence or pool block) of this
    // lane's boxes of tile t: [0..1] this CTA's rows, [2..3] the peer's. Paged,
    // a tile's table entries are requested one tile ahead (`fetch`) and checked
    // when used (`check`), so the lookups wait on nothing.
    struct Coords {
      int c1[4], c2[4], ti[4];
    };
    auto fetch = [&](int t) -> Coords {
      Coords c;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool own = i < 2;
        const int x = lane + 32 * (i & 1);
        const int row_base = k0 + t * kKeys + kOwn * (own ? half : 1 - half);
        c.c1[i] = row_base;  // contiguous: rows past the cache's capacity read as zeros
        c.c2[i] = b;
        c.ti[i] = -1;
        if (!p.tables || x >= (own ? C::kNB : C::kCBV) * per) continue;
        const int row0 = row_base + (x % per) * br;
        c.c1[i] = row0 % p.bs;
        c.c2[i] = p.num_blocks;  // a block past the sequence loads from past the end of the pool: zeros
        if (row0 / p.bs < p.mbps && row0 < len) {
          c.ti[i] = row0 / p.bs;
          c.c2[i] = __ldg(p.tables + (size_t)b * p.mbps + c.ti[i]);
        }
      }
      return c;
    };
    auto check = [&](Coords& c) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (c.ti[i] >= 0 && (c.c2[i] < 0 || c.c2[i] >= p.num_blocks)) {  // an entry out of range: flagged, zeros
          raise_error(p.err, kErrBounds);
          c.c2[i] = p.num_blocks;
        }
    };
    // load one part of tile t once its stage is free; false once a wait gave up
    auto load_part = [&](int t, bool own, const int* c1, const int* c2) -> bool {
      const int nb = own ? C::kNB : C::kCBV;
      const int nbox = whole ? 1 : nb * per;
      const int stages = own ? kStagesR : kStagesV;
      const int st = t % stages;
      uint64_t* full = own ? &bars->r_full[st] : &bars->v_full[st];
      if (t >= stages) {  // the stage is free once PV_{t - stages} is done
        // (o_done[u % kStagesR] completes once per PV_u, u = t - stages; its next
        // phase, PV_{u + kStagesR}, needs a tile this loop has not loaded yet)
        const int u = t - stages;
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(&bars->o_done[u % kStagesR], (u / kStagesR) & 1, bars, p.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      }
      if (lane == 0) mbar_arrive_expect_tx(full, nb * C::kRBlk);
      __syncwarp();
      unsigned char* dst = smem + (own ? C::kOffR + st * C::kStageR : C::kOffV + st * C::kStageV);
      if (whole) {
        if (lane == 0) tc::tma_load_4d(dst, own ? &tm_r : &tm_v, 0, c1[0], own ? 0 : half * C::kCBV, c2[0], full);
      } else {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int x = lane + 32 * u;
          if (x >= nbox) continue;
          const int cb = x / per;                        // block within the part
          const int g = own ? cb : half * C::kCBV + cb;  // the row's column block
          tc::tma_load_4d(dst + cb * C::kRBlk + (x % per) * br * 128, &tm_r, 0, c1[u], g, c2[u], full);
        }
      }
      __syncwarp();
      if (own)
        last_r[st] = t;
      else
        last_v[st] = t;
      return true;
    };
    if (whole) {
      // one box per part: lane 0 runs the loop alone
      if (lane == 0) {
        const bool skip0 = p.debug_withhold && half == 1;  // test hook: tile 0 is never requested
        // paged: the pool block holding a part's 32 rows starting at `row` (bs
        // >= 32, so one block holds them); a part past the sequence loads from
        // past the end of the pool (zeros). Requested one tile ahead.
        struct Entry {
          int e;        // sequence (contiguous) or pool block
          bool looked;  // read from the table (and so to be checked)
        };
        auto entry = [&](int row) -> Entry {
          if (!p.tables) return Entry{b, false};
          const int ti = row / p.bs;
          if (ti < p.mbps && row < len) return Entry{__ldg(p.tables + (size_t)b * p.mbps + ti), true};
          return Entry{p.num_blocks, false};
        };
        // checked when used: an entry out of range is flagged and reads zeros
        auto use = [&](Entry x) {
          if (x.looked && (x.e < 0 || x.e >= p.num_blocks)) {
            raise_error(p.err, kErrBounds);
            return p.num_blocks;
          }
          return x.e;
        };
        auto part_row = [&](int t, bool own) { return k0 + t * kKeys + kOwn * (own ? half : 1 - half); };
        auto issue_r = [&](int t, Entry x) -> bool {  // this CTA's rows of tile t
          const int sr = t % kStagesR;
          // a stage is free once PV_{t - stages} is done (o_done completes once per PV)
          if (t >= kStagesR && !wait_or_abort(&bars->o_done[(t - kStagesR) % kStagesR], ((t - kStagesR) / kStagesR) & 1,
                                              bars, p.err))
            return false;
          const int c1 = p.tables ? part_row(t, true) % p.bs : part_row(t, true);
          mbar_arrive_expect_tx(&bars->r_full[sr], C::kStageR);
          tc::tma_load_4d(smem + C::kOffR + sr * C::kStageR, &tm_r, 0, c1, 0, use(x), &bars->r_full[sr]);
          last_r[sr] = t;
          return true;
        };
        auto issue_v = [&](int t, Entry x) -> bool {  // the peer's rows of tile t, this CTA's value blocks
          const int sv = t % kStagesV;
          if (t >= kStagesV && !wait_or_abort(&bars->o_done[(t - kStagesV) % kStagesR], ((t - kStagesV) / kStagesR) & 1,
                                              bars, p.err))
            return false;
          const int c1 = p.tables ? part_row(t, false) % p.bs : part_row(t, false);
          mbar_arrive_expect_tx(&bars->v_full[sv], C::kStageV);
          tc::tma_load_4d(smem + C::kOffV + sv * C::kStageV, &tm_v, 0, c1, half * C::kCBV, use(x), &bars->v_full[sv]);
          last_v[sv] = t;
          return true;
        };
        // The R ring runs one tile ahead of the V ring: R_0 and R_1 go out at
        // once, V_0 and then R_2 onwards land over the Q_abs staging area, so
        // they wait for q_full. Table entries are requested a step ahead.
        Entry x_r = entry(part_row(0, true)), x_v = entry(part_row(0, false));
        bool ok = skip0 || issue_r(0, x_r);
        x_r = entry(part_row(min(1, n_t - 1), true));
        for (int t = 0; ok && t < n_t; ++t) {
          const Entry r_next = x_r, v_cur = x_v;  // R_{t+1}, V_t
          x_r = entry(part_row(min(t + 2, n_t - 1), true));
          x_v = entry(part_row(min(t + 1, n_t - 1), false));
          if (t + 1 < n_t && !issue_r(t + 1, r_next)) break;
          if (t == 0 && !wait_or_abort(&bars->q_full, 0, bars, p.err)) break;
          if (!(skip0 && t == 0) && !issue_v(t, v_cur)) break;
        }
      }
      __syncwarp();
    } else {
      // the same order as above: this CTA's rows one tile ahead of the peer's
      const bool skip0 = p.debug_withhold && half == 1;  // test hook: tile 0 is never requested
      Coords cur = fetch(0);                     // tile t
      Coords nxt = fetch(min(1, n_t - 1));       // tile t + 1, in flight
      check(cur);
      bool ok = skip0 || load_part(0, true, cur.c1, cur.c2);
      for (int t = 0; ok && t < n_t; ++t) {
        const Coords nn = fetch(min(t + 2, n_t - 1));  // in flight during this step's waits
        check(nxt);
        if (t + 1 < n_t && !load_part(t + 1, true, nxt.c1, nxt.c2)) break;
        if (t == 0) {
          bool g = true;
          if (lane == 0) g = wait_or_abort(&bars->q_full, 0, bars, p.err);
          if (!__shfl_sync(0xffffffffu, g, 0)) break;
        }
        if (!(skip0 && t == 0) && !load_part(t, false, cur.c1 + 2, cur.c2 + 2)) break;
        cur = nxt;
        nxt = nn;
      }
    }
    if (lane == 0) {  // never exit with a load in flight
      if (!mbar_wait(&bars->q_full, 0)) raise_error(p.err, kErrTimeout);
      if (!mbar_wait(&bars->q_stage, 0)) raise_error(p.err, kErrTimeout);
      for (int s = 0; s < kStagesR; ++s)
        if (last_r[s] >= 0 && !mbar_wait(&bars->r_full[s], (last_r[s] / kStagesR) & 1)) raise_error(p.err, kErrTimeout);
      for (int s = 0; s < kStagesV; ++s)
        if (last_v[s] >= 0 && !mbar_wait(&bars->v_full[s], (last_v[s] / kStagesV) & 1)) raise_error(p.err, kErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA issuer =================
    // The warp runs the loop converged, every decision warp-uniform, and an
    // elected lane issues the MMAs two at a time, and each commit: a converged
    // warp keeps the tensor core at its rate on these short (N = 32) MMAs, a lone
    // lane does not (the 36 score MMAs: ~1,750 cycles of issue from one lane,
    // ~1,100 from the warp; the whole call with one MMA per election 59.1 us,
    // two 55.9, four 58.7).
    {
      const uint32_t idS = tc::idesc_bf16_f32(kHeads, kOwn, false);
      const uint32_t idO = tc::idesc_bf16_f32(kHeads, C::kDVH, true);
      constexpr uint64_t kHiK = tc::desc_sw128_hi(0, 1024);  // K-major: 8-row groups 1024 bytes apart
      // V: MN-major, 8-row groups 1024 bytes apart, 64-column blocks one 32-row block apart
      constexpr uint64_t kHiV = tc::desc_sw128_hi(C::kRBlk, 1024);
      // P: K-major without swizzle, 8-key columns kPCol apart, 8-head groups 128 bytes apart
      constexpr uint64_t kHiP = tc::desc_plain_hi(C::kPCol, 128);
      const uint64_t dQ = kHiK | tc::desc_addr(smem + C::kOffQ);
      const uint64_t dR0 = kHiK | tc::desc_addr(smem + C::kOffR);
      // values of this CTA's keys: its value blocks of the R stage; of the peer's keys: the V stage
      const uint64_t dVo0 = kHiV | tc::desc_addr(smem + C::kOffR + half * C::kCBV * C::kRBlk);
      const uint64_t dVp0 = kHiV | tc::desc_addr(smem + C::kOffV);
      const uint64_t dP0 = kHiP | tc::desc_addr(smem + C::kOffR + (1 - half) * C::kCBV * C::kRBlk);
      const uint32_t tO = tmem + C::kColO, tS = tmem + C::kColS, tQ = tmem + C::kColQ;
      auto issue_s = [&](int t) {  // S = Q_abs (this CTA's 32 rows of R_t)^T
        const int st = t % kStagesR;
        tc::fence_after_sync();
        const uint64_t dR = dR0 + (uint64_t)((st * C::kStageR) >> 4);
#pragma unroll
        for (int k0 = 0; k0 < C::kW / 16; k0 += 2) {
          if (tc::elect_one()) {
#pragma unroll
            for (int kk = k0; kk < k0 + 2; ++kk) {
              const int g = kk / 4, step = kk % 4;  // column block, 16-column step inside it
              const uint32_t ar = g * C::kRBlk + step * 32;
              if (g < C::kQT)  // Q_abs from TMEM: 16 columns = 8 TMEM columns
                tc::mma_f16_ts(tS, tQ + g * 32 + step * 8, dR + (ar >> 4), idS, kk > 0);
              else
                tc::mma_f16_ss(tS, dQ + (((g - C::kQT) * C::kQBlk + step * 32) >> 4), dR + (ar >> 4), idS, kk > 0);
            }
          }
          __syncwarp();
        }
        if (tc::elect_one()) tc::mma_commit(&bars->s_full);
        __syncwarp();
      };
      auto issue_pv = [&](int t) {  // O += P_t R_t[:, value half], 16 keys per instruction
        const int sr = t % kStagesR, sv = t % kStagesV;
        tc::fence_after_sync();
        const uint64_t dP = dP0 + (uint64_t)((sr * C::kStageR) >> 4);
        const uint64_t dVo = dVo0 + (uint64_t)((sr * C::kStageR) >> 4);
        const uint64_t dVp = dVp0 + (uint64_t)((sv * C::kStageV) >> 4);
#pragma unroll
        for (int k0 = 0; k0 < kKeys / 16; k0 += 2) {
          if (tc::elect_one()) {
#pragma unroll
            for (int kk = k0; kk < k0 + 2; ++kk) {
              // keys 16kk .. 16kk + 15 of the tile are rows of CTA kk / 2
              const uint64_t dV = (kk / 2 == half ? dVo : dVp) + (uint64_t)(((kk % 2) * 16 * 128) >> 4);
              tc::mma_f16_ss(tO, dP + (uint64_t)((kk * 2 * C::kPCol) >> 4), dV, idO, (t > 0 || kk > 0));
            }
          }
          __syncwarp();
        }
        if (tc::elect_one()) {
          tc::mma_commit(&bars->o_done[sr]);
        }
        __syncwarp();
      };
      bool ok = warp_wait(&bars->q_full, 0, bars, p.err);
      // S_t needs this CTA's rows of tile t and S_{t-1} read (one S buffer); PV_t
      // needs both halves of P_t and the peer's rows. Each barrier is probed for its phases in order
      // and cannot run two phases ahead. A step is taken once every lane has
      // seen its barrier complete.
      int next_s = 0, next_pv = 0;
      long long idle_since = clock64();
      while (ok && next_pv < n_t) {
        bool progressed = false;
        // PV first: its completion frees a ring stage and a P tile
        const bool pv_ready = next_pv < next_s && mbar_test_parity_nb(&bars->p_full[next_pv & 1], (next_pv >> 1) & 1) &&
                              mbar_test_parity_nb(&bars->v_full[next_pv % kStagesV], (next_pv / kStagesV) & 1);
        if (__all_sync(0xffffffffu, pv_ready)) {
          issue_pv(next_pv++);
          progressed = true;
        }
        const bool s_ready = next_s < n_t &&
                             mbar_test_parity_nb(&bars->r_full[next_s % kStagesR], (next_s / kStagesR) & 1) &&
                             (next_s == 0 || mbar_test_parity_nb(&bars->s_free, (next_s - 1) & 1));
        if (__all_sync(0xffffffffu, s_ready)) {
          issue_s(next_s++);
          progressed = true;
        }
        if (progressed) {
          idle_since = clock64();
        } else {
          // lane 0's view decides for the warp
          const int stop = __shfl_sync(0xffffffffu, aborted(bars) ? 1 : (clock64() - idle_since > kWaitLimitCycles ? 2 : 0), 0);
          if (stop == 2 && lane == 0) abort_all(bars, p.err);
          if (stop) ok = false;
        }
      }
      // every MMA issued above has completed before TMEM is released
      if (tc::elect_one()) tc::mma_commit(&bars->mma_final);
      __syncwarp();
      if (lane == 0 && !mbar_wait(&bars->mma_final, 0)) raise_error(p.err, kErrTimeout);
      __syncwarp();
    }
  } else {
    // ================= softmax: thread t owns head h0 + t =================
    const int r = warp * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    const int h = h0 + r;
    const bool mine = h < p.H;
    // ---- the head's first kQT blocks of Q_abs into TMEM (column c holds
    // elements 2c and 2c+1), from their copies in the staging area. 128-byte
    // swizzle: piece i (16 bytes) of row r sits at piece i ^ (r % 8) of the
    // row, so a warp's reads of one piece spread over every bank.
    bool alive = warp_wait(&bars->q_stage, 0, bars, p.err);
    if (alive) {
      const uint32_t qrow = smem_u32(smem + C::kOffStage) + r * 128;
#pragma unroll
      for (int g = 0; g < C::kQT; ++g) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          ld_shared_v4(qrow + g * C::kQBlk + ((i ^ (r & 7)) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        tc::tmem_st_32x32b_x32(tmem + lane_addr + C::kColQ + g * 32, w);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_full);  // the staging area may be refilled
    }
    const float qs = p.qscale;
    const float th = kRescaleLog2 / qs;
    const float2 qs2 = make_float2(qs, qs);
    const uint32_t tS = tmem + lane_addr + C::kColS;
    float m_ref = -INFINITY, l_own = 0.f;  // l_own: the row sum of this CTA's p
    for (int t = 0; alive && t < n_t; ++t) {
      const int x = t & 1;
      if (!warp_wait(&bars->s_full, t & 1, bars, p.err)) {
        alive = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t sv[kOwn];
      tc::tmem_ld_32x32b_x32(tS, sv);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free);
      // rows of the pair's tile the heads see: this CTA's 32 and the peer's 32
      const int kt = k0 + t * kKeys;
      const int valid_own = max(0, min(kOwn, k1 - (kt + kOwn * half)));
      const int valid_peer = max(0, min(kOwn, k1 - (kt + kOwn * (1 - half))));
      if (valid_own < kOwn) {
#pragma unroll
        for (int e = 0; e < kOwn; ++e)
          if (e >= valid_own) sv[e] = __float_as_uint(-INFINITY);
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < kOwn; e += 2)
        mx4[(e >> 1) & 3] = fmax3(mx4[(e >> 1) & 3], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
      const float mx_own = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // ---- the tile max over both CTAs' rows: trade maxima with the peer's warp.
      // The peer copies its P_t columns here only once it has these maxima, and
      // they complete on p_full[x] like its P_{t-2} columns did: so the maxima
      // go out only after P_{t-2} is complete here (long since, in practice).
      if (t >= 2 && !warp_wait(&bars->p_full[x], ((t - 2) >> 1) & 1, bars, p.err)) {
        alive = false;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&bars->m_full[warp][x], 32 * 4);
      st_async_b32(peer_addr(mbuf + x * kHeads + r, peer), __float_as_uint(mx_own),
                   peer_addr(&bars->m_full[warp][x], peer));
      if (!warp_wait_cluster(&bars->m_full[warp][x], (t >> 1) & 1, bars, p.err)) {
        alive = false;
        break;
      }
      const float mx = fmaxf(mx_own, ld_shared_f32(smem_u32(mbuf + x * kHeads + r)));
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
          if (!warp_wait(&bars->o_done[(t - 1) % kStagesR], ((t - 1) / kStagesR) & 1, bars, p.err)) {
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
          l_own *= f;
        }
      }
      // p = 2^(s*qs - m*qs) as bf16 pairs, and the fp32 sum of exactly these p
      const float mq = m_ref * qs;
      const float2 nmq2 = make_float2(-mq, -mq);
      uint32_t pw[kOwn / 2];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kOwn / 2; ++i) {
        const float2 xv = __ffma2_rn(make_float2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), qs2, nmq2);
        pw[i] = ex2_bf16x2(pack_bf16(xv.x, xv.y));
        add_bf16x2(ls[(i & 1) * 2], ls[(i & 1) * 2 + 1], pw[i]);
      }
      l_own += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      unsigned char* rstage = smem + C::kOffR + (t % kStagesR) * C::kStageR;
      if (valid_own < kOwn || valid_peer < kOwn) {
        // value rows of keys at or past seq_len, in this CTA's rows (its value
        // blocks; S_t, their other reader, is done) and in the peer rows' V
        // stage (once it has landed): zero them so that 0 * (whatever the cache
        // holds) cannot be NaN
        unsigned char* vstage = smem + C::kOffV + (t % kStagesV) * C::kStageV;
        if (valid_peer < kOwn && !warp_wait(&bars->v_full[t % kStagesV], (t / kStagesV) & 1, bars, p.err)) {
          alive = false;
          break;
        }
        const int n_own = (kOwn - valid_own) * C::kCBV * 8;  // 16-byte chunks: 8 per row and block
        const int n_all = n_own + (kOwn - valid_peer) * C::kCBV * 8;
        for (int i = r; i < n_all; i += kHeads) {
          const bool o = i < n_own;
          const int j = o ? i : i - n_own;
          const int row = (o ? valid_own : valid_peer) + j / (C::kCBV * 8), blk = (j / 8) % C::kCBV, ch = j % 8;
          unsigned char* base = o ? rstage + (half * C::kCBV + blk) * C::kRBlk : vstage + blk * C::kRBlk;
          *reinterpret_cast<uint4*>(base + row * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // ---- this CTA's 32 keys of P_t: 8-key columns 4 half .. 4 half + 3 of
      // the tile's P, which sits in the R stage over the other half's value
      // blocks (only S_t read them, and S_t is done; the peer's copy of its
      // columns comes after it has this CTA's maxima, sent after S_t too). Each
      // head's 16 bytes at row offset 16 r; then the warp's rows of those
      // columns (512 bytes each) into the same place of the peer's P, which
      // sits over this CTA's value blocks there.
      unsigned char* pt = rstage + (1 - half) * C::kCBV * C::kRBlk;
      unsigned char* pt_peer = rstage + half * C::kCBV * C::kRBlk;
      const uint32_t pbase = smem_u32(pt);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        st_shared_v4(pbase + (4 * half + i) * C::kPCol + r * 16, pw[4 * i], pw[4 * i + 1], pw[4 * i + 2],
                     pw[4 * i + 3]);
      tc::fence_async_smem();  // P and the zeroed rows visible to the tensor cores and the bulk copies
      __syncwarp();
      if (lane < 4) {  // one 512-byte copy per lane: the four in one instruction
        const int off = (4 * half + lane) * C::kPCol + warp * 32 * 16;
        bulk_copy_to_peer(peer_addr(pt_peer + off, peer), pt + off, 32 * 16, peer_addr(&bars->p_full[x], peer));
      }
      if (lane == 0) {
        if (warp == 0)
          mbar_arrive_expect_tx(&bars->p_full[x], kHeads * kOwn * 2);  // the peer's half, incoming
        else
          mbar_arrive(&bars->p_full[x]);
      }
    }
    // ---- the last PV (its commit covers every earlier MMA); the pair's row sum
    bool have_o = alive;
    if (have_o) {
      have_o = warp_wait(&bars->o_done[(n_t - 1) % kStagesR], ((n_t - 1) / kStagesR) & 1, bars, p.err);
      tc::fence_after_sync();
    }
    float l_run = 0.f;
    if (have_o) {
      if (lane == 0) mbar_arrive_expect_tx(&bars->l_full[warp], 32 * 4);
      st_async_b32(peer_addr(lbuf + r, peer), __float_as_uint(l_own), peer_addr(&bars->l_full[warp], peer));
      have_o = warp_wait_cluster(&bars->l_full[warp], 0, bars, p.err);
      if (have_o) l_run = l_own + ld_shared_f32(smem_u32(lbuf + r));  // the same sum on both sides
    }
    // ---- O out. Each thread holds its head's row of this CTA's value half in
    // TMEM; 32 columns at a time, the warp moves its 32 rows through a padded
    // shared-memory buffer (row stride 33 words: no bank conflict either way)
    // so that each store writes one row's 32 consecutive columns. The buffer
    // lies in the R ring, free now: every tile is consumed and the last PV done.
    // One sequence split: O / l as bf16; otherwise (m, l, O) in fp32.
    float* stage = reinterpret_cast<float*>(smem + C::kOffR) + warp * 32 * 33;
    const float inv = (have_o && l_run > 0.f) ? 1.f / l_run : 0.f;
    if (n_split > 1 && mine && half == 0) {
      float* P = p.partial + (((size_t)b * p.H + h) * p.max_splits + split) * (DC + 2);
      P[0] = have_o ? m_ref * qs : -INFINITY;
      P[1] = have_o ? l_run : 0.f;
    }
    const int h_w = h0 + warp * 32;  // the warp's first head
    const int nrows = min(32, p.H - h_w);  // rows of this warp that are heads
    // row i of the warp at dst0 + i * row_stride (elements), this lane's column within the chunk
    const size_t row0 = (size_t)b * p.H + h_w;
    const size_t row_stride = n_split == 1 ? (size_t)DC : (size_t)p.max_splits * (DC + 2);
    __nv_bfloat16* out0 = p.out + row0 * DC + half * C::kDVH + lane;
    float* part0 = p.partial + (row0 * p.max_splits + split) * (DC + 2) + 2 + half * C::kDVH + lane;
    float inv_r[32];  // each row's 1 / l (one sequence split)
#pragma unroll
    for (int i = 0; i < 32; ++i) inv_r[i] = __shfl_sync(0xffffffffu, inv, i);
#pragma unroll 1
    for (int c = 0; c < C::kDVH / 32; ++c) {
      uint32_t o[32];
      tc::tmem_ld_32x32b_x32(tmem + lane_addr + C::kColO + c * 32, o);
      tc::tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) stage[lane * 33 + e] = __uint_as_float(o[e]);
      __syncwarp();
      float v[32];  // row i's column c * 32 + lane: every read first, then the stores
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = stage[i * 33 + lane];
      __syncwarp();  // the buffer is refilled for the next chunk
      if (n_split == 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < nrows) out0[i * row_stride + c * 32] = __float2bfloat16_rn(v[i] * inv_r[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < nrows) part0[i * row_stride + c * 32] = v[i];
      }
    }
  }

  grid_dep_launch();  // the split combine may start launching on freed SMs
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer's last accesses to this CTA's shared memory are done
  tc::fence_after_sync();
  if (aborted(bars)) {
    // after a wait gave up, a store or copy the peer issued into this CTA just
    // before it stopped may still be landing: give it time (bounded) before the
    // shared memory is released
    const long long t0 = clock64();
    while (clock64() - t0 < 200000) {
    }
  }
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

// The same rows of w = 64 nb elements seen as [outer][row][column block][64]:
// dimensions 64, rows, nb, outer with byte strides 2w (a row), 128 (a block),
// 2w rows (an outer index). A box of box_rows rows x box_blk blocks lands in
// shared memory block after block, box_rows x 128 bytes each, 128-byte swizzle;
// rows past the tensor read as zeros.
bool make_blocks_map(CUtensorMap* m, const void* base, int w, uint64_t rows, uint64_t outer, uint32_t box_rows,
                     uint32_t box_blk) {
  const uint64_t dims[4] = {64, rows, (uint64_t)(w / 64), outer};
  const uint64_t strides[3] = {(uint64_t)w * 2, 128, (uint64_t)w * 2 * rows};
  const uint32_t box[4] = {64, box_rows, box_blk, 1};
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
  CUtensorMap tq, tr, tv;
  // q_abs [B, H, 576]: box of 128 heads
  if (!make_rows_map(&tq, q_abs, C::kW, (uint64_t)H, (uint64_t)B, kHeads)) return cudaErrorInvalidValue;
  // latent [B, max_len, 576] or pool [num_blocks, bs, 576]: boxes of one CTA's
  // 32 rows of a tile, all blocks (tr) or a value half (tv); a pool of 8- or
  // 16-row blocks: boxes of one pool block x one column block (tr; tv unused)
  const uint64_t rows = tables ? (uint64_t)bs : (uint64_t)max_len;
  const uint64_t outer = tables ? (uint64_t)num_blocks : (uint64_t)B;
  const bool whole = !tables || bs >= kOwn;
  const uint32_t br = whole ? kOwn : (uint32_t)bs;
  if (!make_blocks_map(&tr, latent, C::kW, rows, outer, br, whole ? C::kNB : 1) ||
      !make_blocks_map(&tv, latent, C::kW, rows, outer, br, whole ? C::kCBV : 1))
    return cudaErrorInvalidValue;
  if (tables) max_len = mbps * bs;
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
  p.q_abs = static_cast<const __nv_bfloat16*>(q_abs);
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
  return cudaLaunchKernelEx(&cfg, mla_absorbed_tc_kernel<512, 64>, tq, tr, tv, p);
}

}  // namespace gqa
