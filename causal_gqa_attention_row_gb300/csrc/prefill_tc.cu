// prefill_tc.cu -- causal prefill on the tcgen05 tensor cores (bf16; (d_k, d_v) = (64, 64),
// (128, 128) or (192, 128)).
//
// The operation (kopitiam-runtime src/attention.rs, `attention_forward` and
// `causal_mask`): row i of sequence b, query head h, sits at position
// offset_b + i and attends to keys 0..=offset_b + i of KV head h / G with
// softmax(scale * q.k); everything else weighs exactly zero.
//
// One CTA = one (sequence, query head, 128-row query tile); CTAs are ordered
// longest-first (the causal work of a tile grows with its index). Roles, one
// warpgroup each, with registers moved from the control warpgroup to the two
// softmax warpgroups (setmaxnreg: 72 and 216 per thread from 168 at launch):
//   warps 0-3   softmax warpgroup 0: key tiles 0, 2, 4, ...
//   warps 4-7   softmax warpgroup 1: key tiles 1, 3, 5, ...
//   warp 8      initialises the barriers; TMA producer of Q (once) and of the
//               128-key K tiles (a four-stage ring at d_k = 64, two-stage for
//               wider heads; 128-byte swizzle, the layout the MMA reads)
//   warps 9, 10 one thread each issues the tcgen05.mma of one softmax warpgroup
//               (warp 9 also allocates and frees TMEM)
//   warp 11     TMA producer of the V tiles (ring as for K)
// Warpgroup w owns, in tensor memory (TMEM), S_w = Q K^T (M=128, N=128, K=d_k;
// 128 columns), P_w (the bf16 probabilities, two per 32-bit column; 64 columns)
// and O_w += P_w V (M=128, N=d_v, K=128, A read from TMEM; d_v columns). At
// d_v = 64 the three are separate (S 2 x 128 + O 2 x 64 + P 2 x 64 = 512
// columns); at d_v = 128 P_w sits over the first 64 columns of S_w (S 2 x 128 +
// O 2 x 128), so the MMA thread issues the next S into S_w only once the PV that
// reads P_w is done. P never passes through shared memory, whose bandwidth is
// left to the TMA tiles and the MMAs' reads of Q, K and V. A row of d elements
// is d / 64 blocks of 64 columns, each in the 128-byte swizzle (one TMA box). The
// softmax threads form p with fp32 exponentials, keep the fp32 row sum of these
// p, and round P to bf16 for the PV product. Thread t of a warpgroup owns query
// row t (TMEM lane t).
//
// Pipeline per warpgroup and key tile j: the softmax threads load their S_j row
// into registers and release S_w at once, so the MMA thread issues S_{j+2}
// while the exponentials of tile j are still being computed. P_j goes into P_w
// once PV_{j-2} (issued a whole tile earlier) has read the previous one: at
// d_v = 64 all of it after the exponentials, which overlap that PV; at d_v = 128
// (S_w holds S_j only once that PV is done) chunk by chunk as it is formed, its
// first half (keys 0-63) signalled on a barrier of its own so that the MMA
// thread issues that half of PV_j while the rest is formed. K and V have rings
// of their own: a K stage is free as soon as its S MMA is done,
// a V stage once its PV is. At d_k = 64 they run four tiles ahead, so the load of
// K_{j+4} has a whole tile-period before S_{j+4} needs it; for wider heads (tiles
// two or three times the size) two, which the later issue of S leaves enough.
//
// Softmax with lazy rescaling: p = 2^((s - m) * scale * log2 e) against a
// reference max m that only moves when a score exceeds it by more than 2^8 in
// p, which keeps every p <= 256 and leaves O / l unchanged. Each tile's row max
// is taken first; in the rare case it passes the reference by the threshold,
// the reference moves and O_w (in TMEM, after every PV issued so far has
// completed) and l are rescaled. Keys past the row's position (only in tiles
// that cross the diagonal) weigh exactly zero. At the end the two warpgroups
// exchange their (m, l), each merges half of the columns of the two partial O
// rows into bf16 in shared memory (over the Q tile), and one TMA store writes
// the output tile.
//
// Launches use programmatic stream serialization: a CTA initialises its
// barriers, allocates TMEM and prefetches its tensor maps before waiting for
// the previous kernel in the stream (griddepcontrol.wait), and lets the next
// launch start once it is set up, so back-to-back launches overlap one's set-up
// with the other's tail.

#include <atomic>
#include "tc_ptx.cuh"
#include "tmap.h"

namespace gqa {
namespace {

constexpr int kBM = 128;   // query rows per tile
constexpr int kBN = 128;   // keys per tile
constexpr int kWG = 2;     // softmax warpgroups
constexpr int kThreads = (kWG + 1) * 128;  // two softmax warpgroups + one control warpgroup
constexpr int kProducerWarp = 8, kMmaWarp0 = 9, kProducerVWarp = 11;
// Registers per thread: 168 at launch (384 threads); the control warpgroup
// gives up 96 per thread and the softmax warpgroups take 48 more:
// 128 * 72 + 256 * 216 = 384 * 168. (88 / 208 measured the same at d = 64 and
// d = 128 and up to 1% slower for the arms, the MLA widths and the paged chunks;
// 56 / 224 the same as 72 / 216.)
constexpr int kLaunchRegs = 168, kCtrlRegs = 72, kSoftmaxRegs = 216;
static_assert(128 * kCtrlRegs + kWG * 128 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split over budget");
constexpr int kBlk = kBM * 128;  // 16 KiB: 128 rows of one 64-column block
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kTabEntries = 4096;  // paged: the CTA's block-table entries
constexpr int kMaxStages = 4;

// Sizes and maps of the kernel for head widths DK (Q, K) and DV (V, out).
template <int DK, int DV>
struct Cfg {
  static constexpr int kCBK = DK / 64, kCBV = DV / 64;  // 64-column blocks of a Q/K row, of a V/out row
  static constexpr int kTileK = kCBK * kBlk;            // one Q or K tile (128 rows)
  static constexpr int kTileV = kCBV * kBlk;            // one V or output tile
  static constexpr bool kAlias = DV > 64;               // P_w over the first 64 columns of S_w
  // rings: stage s only ever holds key tiles of warpgroup s % 2
  static constexpr int kStagesK = DK > 64 ? 2 : 4, kStagesV = DK > 64 ? 2 : 4;
  static_assert(kStagesK % kWG == 0 && kStagesV % kWG == 0 && kStagesK <= kMaxStages && kStagesV <= kMaxStages,
                "ring stages shared between warpgroups");
  static_assert(DV <= DK, "the output tile is staged over Q");
  // TMEM columns of S_w, O_w and P_w
  __host__ __device__ static constexpr uint32_t col_s(int w) { return kAlias ? (128 + DV) * w : 128 * w; }
  __host__ __device__ static constexpr uint32_t col_o(int w) { return kAlias ? (128 + DV) * w + 128 : 256 + 64 * w; }
  __host__ __device__ static constexpr uint32_t col_p(int w) { return kAlias ? (128 + DV) * w : 384 + 64 * w; }
  static_assert(col_o(kWG - 1) + DV <= kTmemCols && col_p(kWG - 1) + 64 <= kTmemCols, "TMEM map");
  // shared-memory map (from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTileK;                             // K ring
  static constexpr int kOffV = kOffK + kStagesK * kTileK;          // V ring
  static constexpr int kOffTab = kOffV + kStagesV * kTileV;        // paged: block-table entries
  static constexpr int kOffBar = kOffTab + kTabEntries * 4;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;          // + alignment slack
  // At the end, once every MMA is done: the output tile over Q, and warpgroup
  // w's row max and sum over K stage w (which only ever held warpgroup w's tiles).
  static constexpr int kOffOut = kOffQ;
  static constexpr int kOffML = kOffK;
  static_assert(kSmemBytes <= 232448, "over the 227 KiB a CTA may use");
};

struct TcParams {
  int B, S, H, Hkv, G, S_kv, n_qtiles;  // S_kv: keys a sequence can hold (the pool's capacity when paged)
  const int32_t* offsets;
  // paged K/V (tables != NULL): [num_blocks, Hkv, bs, d] pools, row j of
  // sequence b in block tables[b * mbps + j / bs], slot j % bs; bs divides 128
  const int32_t* tables;
  int mbps, bs, num_blocks;
  __nv_bfloat16* out;
  float qscale;
  unsigned* err;
  int debug_withhold;  // test hook: the first K tile is never loaded, so its waits run out
  // The arms (the ARMS instantiation): a row at position p sees keys
  // first_visible_key(p, window)..p; a score s (natural units) becomes
  // softcap * tanh(s / softcap) (cap_out = softcap * log2 e, cap_in = scale /
  // softcap applied to the raw q.k), then s + alibi[h] * (key - p); the sink
  // logit sinks[h] joins the softmax denominator only.
  int window;
  float cap_in, cap_out;
  const float* alibi;
  const float* sinks;
};

// First key tile a row at `pos` can see under the window (0 without one).
__device__ __forceinline__ int first_key_tile(int pos, int window) {
  return first_visible_key(pos < 0 ? 0 : pos, window) / kBN;
}

struct Bars {
  uint64_t q_full, k_full[kMaxStages], k_empty[kMaxStages], v_full[kMaxStages], v_empty[kMaxStages];
  uint64_t s_full[kWG], s_free[kWG], p_full[kWG], mma_final[kWG];
  uint64_t p_half[kWG];  // P over S (d_v = 128): keys 0-63 of the warpgroup's P are in place
  uint64_t o_done[kWG];  // every PV of warpgroup w issued so far is done (a phase per PV)
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

template <typename BarsT>
__device__ __forceinline__ bool aborted(BarsT* bars) {
  return *reinterpret_cast<volatile int*>(&bars->abort_flag);
}

// Each probe of an mbarrier suspends a waiter for at most this long. A waiter
// resumes when the phase completes whatever the hint: 20, 200 and 2000 ns gave
// the same times (prefill and absorbed MLA decode, same box), so the hint only
// sets how often a long wait re-checks its time limit and the abort flag.
constexpr uint32_t kWaitHintNs = 20;


// Single-thread wait of the producer and MMA issuers (bounded). A phase that
// has completed is taken at once (the abort flag, a shared-memory load on the
// critical path, is only read when the wait has to wait).
template <typename BarsT>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, BarsT* bars, unsigned* err) {
  if (mbar_test_parity_nb(bar, parity)) return true;
  if (aborted(bars)) return false;
  if (mbar_wait_hint(bar, parity, kWaitHintNs)) return true;
  *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
  raise_error(err, kErrTimeout);
  return false;
}

// Whole-warp version: every lane agrees on the outcome.
template <typename BarsT>
__device__ __forceinline__ bool warp_wait_tc(uint64_t* bar, uint32_t parity, BarsT* bars, unsigned* err) {
  bool ok = mbar_test_parity_nb(bar, parity) || (!aborted(bars) && mbar_wait_hint(bar, parity, kWaitHintNs));
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) {
    *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
    raise_error(err, kErrTimeout);
  }
  return ok;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// p = 2^(s*qs - mq) for two scores: fp32 exponentials (one special-function
// operation per score; the bf16x2 form costs the same per score and needs
// unpacking), added to the fp32 row sum `acc`, and returned rounded to the bf16
// pair that P stores.
__device__ __forceinline__ uint32_t exp2_pair(float s0, float s1, float2 qs2, float2 nmq2, float2& acc) {
  const float2 x = __ffma2_rn(make_float2(s0, s1), qs2, nmq2);
  const float2 e = make_float2(ex2f(x.x), ex2f(x.y));
  acc = __fadd2_rn(acc, e);
  return pack_bf16(e.x, e.y);
}

__device__ __forceinline__ float rcpf(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// The TMA loads of key tile j (128 rows of D) of KV head kvh, sequence b, into
// `dst`, completing a tile's bytes on `bar`: one box per 64-column block of the
// rows, at that block's 16 KiB slot. Contiguous: the tile's 128 rows in one box
// per block. Paged: one box per pool block and column block, addressed through
// the block table (the 128-byte swizzle is a function of the shared address, so
// the pool blocks land exactly where one box would put them). A pool block that
// holds no key below kv_hi, or whose table entry is out of range (flagged),
// loads from past the end of the pool: the TMA engine fills it with zeros.
__device__ __forceinline__ int pool_block(const TcParams& p, int t, int kv_hi, int e) {
  if (t >= p.mbps || t * p.bs >= kv_hi) return p.num_blocks;
  if (e >= 0 && e < p.num_blocks) return e;
  raise_error(p.err, kErrBounds);
  return p.num_blocks;
}

// One thread, the table read from global memory (the first tile, before the
// CTA's shared copy of the table exists).
template <int NCB>
__device__ __forceinline__ void load_kv_tile(const CUtensorMap* tm, unsigned char* dst, uint64_t* bar, int j, int kvh,
                                             int b, const TcParams& p, int kv_hi) {
  mbar_arrive_expect_tx(bar, NCB * kBlk);
  if (!p.tables) {
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) tc::tma_load_4d(dst + cb * kBlk, tm, cb * 64, j * kBN, kvh, b, bar);
    return;
  }
  const int per = kBN / p.bs;
  for (int i = 0; i < per; ++i) {
    const int t = j * per + i;
    const int e = (t < p.mbps && t * p.bs < kv_hi) ? __ldg(p.tables + (size_t)b * p.mbps + t) : 0;
    const int blk = pool_block(p, t, kv_hi, e);
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb)
      tc::tma_load_4d(dst + cb * kBlk + i * p.bs * 128, tm, cb * 64, 0, kvh, blk, bar);
  }
}

// The whole producer warp: lane 0 sets the expected bytes, then each lane issues
// one box (each TMA instruction holds its thread for a few hundred cycles, so
// the boxes of a tile go out side by side), the entries read from the CTA's
// shared copy of its table row.
template <int NCB>
__device__ __forceinline__ void load_kv_tile_warp(const CUtensorMap* tm, unsigned char* dst, uint64_t* bar, int j,
                                                  int kvh, int b, const TcParams& p, int kv_hi, const int* tab,
                                                  int lane) {
  if (lane == 0) mbar_arrive_expect_tx(bar, NCB * kBlk);
  __syncwarp();
  if (!p.tables) {
    if (lane < NCB) tc::tma_load_4d(dst + lane * kBlk, tm, lane * 64, j * kBN, kvh, b, bar);
  } else {
    const int per = kBN / p.bs;  // per * NCB boxes: one lane each while they fit the warp
    for (int x = lane; x < per * NCB; x += 32) {
      const int i = x % per, cb = x / per;
      const int t = j * per + i;
      const int e = (t < p.mbps && t * p.bs < kv_hi) ? tab[t] : 0;  // the shared copy covers every such t
      tc::tma_load_4d(dst + cb * kBlk + i * p.bs * 128, tm, cb * 64, 0, kvh, pool_block(p, t, kv_hi, e), bar);
    }
  }
  __syncwarp();
}

template <int DK, int DV, bool ARMS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const TcParams p) {
  using C = Cfg<DK, DV>;
  constexpr int kTileK = C::kTileK, kTileV = C::kTileV, kStagesK = C::kStagesK, kStagesV = C::kStagesV;
  constexpr int kOffQ = C::kOffQ, kOffK = C::kOffK, kOffV = C::kOffV, kOffTab = C::kOffTab;
  constexpr int kOffOut = C::kOffOut, kOffML = C::kOffML;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item, longest first
  const int per_tile = p.B * p.H;
  const int qt = p.n_qtiles - 1 - (int)(blockIdx.x / per_tile);
  const int rem = (int)(blockIdx.x % per_tile);
  const int h = rem % p.H, b = rem / p.H;
  const int kvh = h / p.G;
  const int i0 = qt * kBM;
  const int rows = min(kBM, p.S - i0);

  if (warp == kProducerWarp && lane == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStagesK; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kStagesV; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int w = 0; w < kWG; ++w) {
      mbar_init(&bars->s_full[w], 1);
      mbar_init(&bars->s_free[w], 4);  // one arrival per softmax warp
      mbar_init(&bars->p_full[w], 4);
      mbar_init(&bars->p_half[w], 4);
      mbar_init(&bars->mma_final[w], 1);
      mbar_init(&bars->o_done[w], 1);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
    tc::prefetch_tmap(&tm_q);
    tc::prefetch_tmap(&tm_k);
    // everything above may overlap the previous kernel in the stream; the loads
    // below read memory it may have written
    grid_dep_wait();
    // Q and the first K tile load while the rest of the CTA sets up
    mbar_arrive_expect_tx(&bars->q_full, kTileK);
#pragma unroll
    for (int cb = 0; cb < C::kCBK; ++cb)
      tc::tma_load_4d(smem + kOffQ + cb * kBlk, &tm_q, cb * 64, h, i0, b, &bars->q_full);
    if (p.debug_withhold) {
      // test hook: K_0 is never requested (nothing is left in flight), so the
      // first wait on it runs into its bound and the CTA gives up
    } else {
      // the first key tile this query tile sees (the window's, with the arms);
      // paged: the tile's table entries are bounded by the offset
      const int off0 = (ARMS || p.tables) && p.offsets ? p.offsets[b] : 0;
      const int jb0 = ARMS ? first_key_tile(off0 + i0, p.window) : 0;
      load_kv_tile<C::kCBK>(&tm_k, smem + kOffK, &bars->k_full[0], jb0, kvh, b, p, off0 + i0 + rows);
    }
  }
  if (warp == kMmaWarp0) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  grid_dep_wait();  // before any thread touches global memory
  const int off = p.offsets ? p.offsets[b] : 0;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  // the next launch in the stream may start setting up on the SMs this grid frees
  grid_dep_launch();

  if (off < 0 || (long long)off + p.S > p.S_kv) {  // the cache cannot hold these rows
    if (threadIdx.x == 0 && qt == p.n_qtiles - 1 && h == 0) raise_error(p.err, kErrBounds);
    for (int idx = threadIdx.x; idx < rows * DV; idx += blockDim.x)
      p.out[(((size_t)b * p.S + i0 + idx / DV) * p.H + h) * DV + idx % DV] = __float2bfloat16_rn(0.f);
    // never exit with a load in flight
    if (warp == kProducerWarp && lane == 0 &&
        !(mbar_wait(&bars->q_full, 0) && (p.debug_withhold || mbar_wait(&bars->k_full[0], 0))))
      raise_error(p.err, kErrTimeout);
    __syncthreads();
    if (warp == kMmaWarp0) tc::tmem_dealloc(tmem, kTmemCols);
    return;
  }
  // key tiles jb .. jb + n_kv - 1: from the first one the tile's first row sees
  // (under the window; 0 without one) to the last row's position. Ring stages,
  // barrier phases and the warpgroup a tile belongs to count tiles from jb.
  const int jb = ARMS ? first_key_tile(off + i0, p.window) : 0;
  const int n_kv = (off + i0 + rows - 1) / kBN + 1 - jb;

  if (warp >= kProducerWarp) {
    regs_dec<kCtrlRegs>();  // the whole control warpgroup, right at the top of its branch
  if (warp == kProducerWarp || warp == kProducerVWarp) {
    // ================= TMA producers: Q and K (warp 8), V (warp 11) =================
    const bool is_k = warp == kProducerWarp;
    // Paged: the two producer warps copy the table entries of the blocks this
    // CTA reads into shared memory first (coalesced, one round trip), so that
    // a tile's lookups never wait on global memory. The launcher takes this
    // kernel only when a table row fits the copy (max_blocks_per_seq <= kTabEntries).
    const int kv_hi = off + i0 + rows;
    const int* tab = nullptr;
    if (p.tables) {
      int* st_tab = reinterpret_cast<int*>(smem + kOffTab);
      const int n_tab = min(min(p.mbps, (kv_hi + p.bs - 1) / p.bs), kTabEntries);
      for (int i = (is_k ? 0 : 32) + lane; i < n_tab; i += 64) st_tab[i] = __ldg(p.tables + (size_t)b * p.mbps + i);
      named_bar_sync(3, 64);
      tab = st_tab;
    }
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    uint64_t* full = is_k ? bars->k_full : bars->v_full;
    uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
    unsigned char* ring = smem + (is_k ? kOffK : kOffV);
    const int tile_bytes = is_k ? kTileK : kTileV;
    const int stages = is_k ? kStagesK : kStagesV;
    if (!is_k && lane == 0) tc::prefetch_tmap(tm);
    int issued_last[kStagesK];
#pragma unroll
    for (int st = 0; st < kStagesK; ++st) issued_last[st] = -1;
    int j = 0;
    if (is_k) {  // Q and K_0 went out before the setup barrier
      issued_last[0] = p.debug_withhold ? -1 : 0;
      j = 1;
    }
    for (; j < n_kv; ++j) {
      const int st = j % stages;
      if (j >= stages) {
        bool w = true;
        if (lane == 0) w = wait_or_abort(&empty[st], ((j / stages) - 1) & 1, bars, p.err);
        if (!__shfl_sync(0xffffffffu, w, 0)) break;
      }
      if (is_k)
        load_kv_tile_warp<C::kCBK>(tm, ring + st * tile_bytes, &full[st], jb + j, kvh, b, p, kv_hi, tab, lane);
      else
        load_kv_tile_warp<C::kCBV>(tm, ring + st * tile_bytes, &full[st], jb + j, kvh, b, p, kv_hi, tab, lane);
      issued_last[st] = j;
    }
    if (lane == 0) {
      // never exit with a load in flight
      if (is_k && !mbar_wait(&bars->q_full, 0)) raise_error(p.err, kErrTimeout);
      for (int st = 0; st < stages; ++st)
        if (issued_last[st] >= 0 && !mbar_wait(&full[st], (issued_last[st] / stages) & 1))
          raise_error(p.err, kErrTimeout);
    }
  } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
    // ================= MMA issuers: warp 9 for warpgroup 0, warp 10 for warpgroup 1 =================
    const int w = warp - kMmaWarp0;
    if (lane == 0) {
      const int n_mine = (n_kv - w + 1) / 2;
      const uint32_t idS = tc::idesc_bf16_f32(kBM, kBN, false);
      const uint32_t idO = tc::idesc_bf16_f32(kBM, DV, true);
      // descriptors: constant high part + (shared address >> 4) in the low bits
      constexpr uint64_t kHi = tc::desc_sw128_hi(0, 1024);
      const uint64_t dQ = kHi | (smem_u32(smem + kOffQ) >> 4);
      const uint64_t dK0 = kHi | (smem_u32(smem + kOffK) >> 4);
      // V of each stage: MN-major, 8-key groups 1024 bytes apart, its 64-column
      // blocks (d_v > 64) a block's 16 KiB apart (the leading byte offset)
      const uint64_t dV0 = tc::desc_sw128_hi(C::kCBV > 1 ? kBlk : 0, 1024) | (smem_u32(smem + kOffV) >> 4);
      const uint32_t dS = tmem + C::col_s(w), dO = tmem + C::col_o(w), tP = tmem + C::col_p(w);
      auto issue_s = [&](int j) -> bool {  // S_w = Q K_j^T
        const int st = j % kStagesK;
        if (!wait_or_abort(&bars->k_full[st], (j / kStagesK) & 1, bars, p.err)) return false;
        tc::fence_after_sync();
        const uint64_t dK = dK0 + (uint64_t)((st * kTileK) >> 4);
        // 16 of the d_k columns per instruction: block kk / 4, 32 bytes per step inside it
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t at = (kk / 4) * kBlk + (kk % 4) * 32;
          tc::mma_f16_ss(dS, dQ + (at >> 4), dK + (at >> 4), idS, kk > 0);
        }
        tc::mma_commit(&bars->s_full[w]);
        tc::mma_commit(&bars->k_empty[st]);  // the K stage is free once S_j is done
        return true;
      };
      bool ok = n_mine > 0 && wait_or_abort(&bars->q_full, 0, bars, p.err) && issue_s(w);
      for (int k = 0; ok && k < n_mine; ++k) {
        const int j = 2 * k + w;
        // d_v = 64: S_{j+2} as soon as the softmax threads have read S_j into registers
        if (!C::kAlias && k + 1 < n_mine) ok = wait_or_abort(&bars->s_free[w], k & 1, bars, p.err) && issue_s(j + 2);
        // P over S (d_v = 128): the first 64 keys' half of PV_j goes out once
        // their P is in place, while the softmax still forms the rest
        if (!ok || !wait_or_abort(C::kAlias ? &bars->p_half[w] : &bars->p_full[w], k & 1, bars, p.err)) break;
        const int st = j % kStagesV;
        if (!wait_or_abort(&bars->v_full[st], (j / kStagesV) & 1, bars, p.err)) break;
        tc::fence_after_sync();
        // O_w += P_j V_j: 16 keys per instruction, P from TMEM (8 columns per 16 keys)
        const uint64_t dV = dV0 + (uint64_t)((st * kTileV) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          if (C::kAlias && kk == kBN / 32) {
            ok = wait_or_abort(&bars->p_full[w], k & 1, bars, p.err);
            if (!ok) break;
            tc::fence_after_sync();
          }
          tc::mma_f16_ts(dO, tP + kk * 8, dV + kk * (2048 >> 4), idO, (k > 0 || kk > 0));
        }
        if (!ok) break;
        tc::mma_commit(&bars->o_done[w]);
        tc::mma_commit(&bars->v_empty[st]);
        // d_v = 128: P_j sits in S_w, so S_{j+2} waits for PV_j (this thread waits
        // every phase of o_done[w] in order)
        if (C::kAlias && k + 1 < n_mine) {
          ok = wait_or_abort(&bars->o_done[w], k & 1, bars, p.err);
          if (ok) {
            tc::fence_after_sync();
            ok = issue_s(j + 2);
          }
        }
      }
      // every MMA issued above has completed before TMEM is released
      tc::mma_commit(&bars->mma_final[w]);
      if (!mbar_wait(&bars->mma_final[w], 0)) raise_error(p.err, kErrTimeout);
    }
  }
  } else {
    // ================= softmax warpgroups =================
    regs_inc<kSoftmaxRegs>();  // both softmax warpgroups, right at the top of their branch
    const int wg = warp >> 2;  // 0 or 1
    const int quarter = warp & 3;                     // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;                // query row within the tile
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int pos = off + i0 + r;                     // absolute position of this row
    // With the arms the scores are moved into log2 units before the max (scale,
    // softcap, ALiBi), so the exponent's multiplier is 1; plain: the raw q.k
    // and the scale folded into the exponent.
    const float qs = ARMS ? 1.f : p.qscale;
    const float th = kRescaleLog2 / qs;
    const float alibi2 = ARMS && p.alibi ? __ldg(p.alibi + h) * kLog2e : 0.f;  // slope in log2 units
    const int lo_key = ARMS ? first_visible_key(pos, p.window) : 0;          // first key this row sees
    const int lo_tile_end = ARMS ? first_visible_key(off + i0 + rows - 1, p.window) : 0;  // window-masked keys end below
    float m_ref = -INFINITY;
    float l_run = 0.f;  // the row sum of this warpgroup's p, against m_ref
    const uint32_t tS = tmem + lane_addr + C::col_s(wg);
    const uint32_t tO = tmem + lane_addr + C::col_o(wg);
    const uint32_t tP = tmem + lane_addr + C::col_p(wg);
    const float2 qs2 = make_float2(qs, qs);
    const int n_mine = (n_kv - wg + 1) / 2;  // key tiles this warpgroup handles
    bool alive = true;
    // Wider heads: warpgroup 1 starts once warpgroup 0 has stored its first P, so
    // that the two form their exponentials half a tile apart rather than side by
    // side (measured: 47.1 -> 44.4 us at d = 128; at d = 64, where the short query
    // tiles dominate, the later start costs more than it saves: 15.75 -> 16.85 us).
    if (C::kAlias && wg == 1 && n_kv > 1) alive = warp_wait_tc(&bars->p_full[0], 0, bars, p.err);
    for (int k = 0; alive && k < n_mine; ++k) {
      const int j = 2 * k + wg;    // counted from the first visible tile jb
      const int j0 = (jb + j) * kBN;  // the tile's first key
      const bool diag = j0 + kBN - 1 > off + i0;  // this tile crosses the diagonal of some row
      const bool below = ARMS && j0 < lo_tile_end;  // ... or holds keys below some row's window
      if (!warp_wait_tc(&bars->s_full[wg], k & 1, bars, p.err)) {
        alive = false;
        break;
      }
      tc::fence_after_sync();
      // ---- the S row into registers; S_w is then free for S_{j+2}
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld_32x32b_x32(tS + c * 32, sv[c]);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[wg]);
      if (ARMS) {  // scale, softcap, ALiBi: log2 units (branches uniform across the CTA, outside the loops)
        // The ALiBi term splits into the tile's part, slope * (j0 - pos), added
        // with the scale or softcap in one packed operation per pair of scores,
        // and the column's part, slope * column, one fma with an immediate.
        const float base = alibi2 * (float)(j0 - pos);  // 0 without ALiBi
        if (p.cap_out > 0.f) {
          // cap * tanh(x) = cap - 2 cap / (e^(2x) + 1), from the special-function
          // unit's 2^x and reciprocal: absolute error near 1e-6 in tanh over the
          // whole range (e^(2x) -> inf gives cap, -> 0 gives -cap), against about
          // 5e-4 for the tanh.approx instruction, which the cap would multiply
          // into the exponent. The rest is packed over pairs of scores.
          const float2 k2 = make_float2(p.cap_in * 2.8853900817779268f, p.cap_in * 2.8853900817779268f);  // 2 log2(e)
          const float2 one2 = make_float2(1.f, 1.f);
          const float2 m2 = make_float2(-2.f * p.cap_out, -2.f * p.cap_out);
          const float2 a2 = make_float2(p.cap_out + base, p.cap_out + base);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 t = __fmul2_rn(make_float2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), k2);
              const float2 dn = __fadd2_rn(make_float2(ex2f(t.x), ex2f(t.y)), one2);
              const float2 y = __ffma2_rn(make_float2(rcpf(dn.x), rcpf(dn.y)), m2, a2);
              sv[c][e] = __float_as_uint(y.x);
              sv[c][e + 1] = __float_as_uint(y.y);
            }
        } else {
          const float2 q2 = make_float2(p.qscale, p.qscale), b2 = make_float2(base, base);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 y =
                  __ffma2_rn(make_float2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), q2, b2);
              sv[c][e] = __float_as_uint(y.x);
              sv[c][e + 1] = __float_as_uint(y.y);
            }
        }
        if (alibi2 != 0.f) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              sv[c][e] = __float_as_uint(fmaf(alibi2, (float)(c * 32 + e), __uint_as_float(sv[c][e])));
        }
      }
      if (diag || below) {  // keys past the row's position, or (arms) below its window, weigh zero
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int key = j0 + c * 32 + e;
            if (key > pos || key < lo_key) sv[c][e] = __float_as_uint(-INFINITY);
          }
      }
      // ---- the tile's row max; the reference moves only past the threshold
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      if (k == 0) {
        m_ref = mx;  // a row's first tile: nothing to rescale
      } else {
        const bool grow = mx > m_ref + th;
        if (__any_sync(0xffffffffu, grow)) {
          float f = 1.f;
          if (grow) {
            f = ex2f((m_ref - mx) * qs);  // 0 while m_ref = -inf
            m_ref = mx;
          }
          // O_w holds every PV issued so far (PV_{k-1} the last): rescale it once
          // done (at d_v = 128 it is: S_k was issued after it)
          if (!C::kAlias && !warp_wait_tc(&bars->o_done[wg], (k - 1) & 1, bars, p.err)) {
            alive = false;
            break;
          }
          tc::fence_after_sync();
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            tc::tmem_ld_32x32b_x32(tO + c * 32, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tc::tmem_st_32x32b_x32(tO + c * 32, o);
          }
          tc::tmem_st_wait();
          l_run *= f;
        }
      }
      // ---- p = 2^(s*qs - m*qs), the fp32 row sum of these p, and P as bf16 pairs
      const float mq = m_ref == -INFINITY ? 0.f : m_ref * qs;  // no visible key yet: all p are 0
      const float2 nmq2 = make_float2(-mq, -mq);
      float2 ls[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) ls[e] = make_float2(0.f, 0.f);
      uint32_t pw[4][16];  // each P pair replaces the two scores it came from: no more registers than S
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int t = 0; t < 16; ++t)
          pw[c][t] = exp2_pair(__uint_as_float(sv[c][2 * t]), __uint_as_float(sv[c][2 * t + 1]), qs2, nmq2, ls[t & 3]);
        // d_v = 128: P goes over S_j's own first columns, already read; each
        // 16-word chunk is stored as soon as it is formed, and once the first
        // two (keys 0-63) are in place their half of PV_j may start
        if (C::kAlias) {
          tc::tmem_st_32x32b_x16(tP + c * 16, pw[c]);
          if (c == 1) {
            tc::tmem_st_wait();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_half[wg]);
          }
        }
      }
      l_run += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
      // ---- d_v = 64: P_w is free once this warpgroup's previous PV has read it.
      // That PV was issued only as this tile began, so the wait comes after the
      // exponentials, which then overlap it. Every phase of o_done[w] is waited
      // for in order, before the next PV can be issued, so the barrier is never
      // two phases ahead of this wait (nor of the rescale's or the final one).
      if (!C::kAlias) {
        if (k >= 1) {
          if (!warp_wait_tc(&bars->o_done[wg], (k - 1) & 1, bars, p.err)) {
            alive = false;
            break;
          }
          tc::fence_after_sync();
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_st_32x32b_x16(tP + c * 16, pw[c]);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();  // this thread's TMEM accesses are done
      __syncwarp();             // ... for every lane of the warp; one lane signals
      if (lane == 0) mbar_arrive(&bars->p_full[wg]);
    }
    // ---- each warpgroup's last PV; the two exchange (m, l), each merges half of
    // the columns of O_0 and O_1 into the output tile, and one TMA store writes it
    bool have_o = alive && n_mine > 0;
    if (have_o) {  // the last PV's commit covers every MMA this warpgroup's thread issued
      have_o = warp_wait_tc(&bars->o_done[wg], (n_mine - 1) & 1, bars, p.err);
      tc::fence_after_sync();
    }
    const float l_sum = l_run;
    float* ml = reinterpret_cast<float*>(smem + kOffML + wg * kTileK);  // K stage wg: consumed by now
    ml[r] = have_o ? m_ref : -INFINITY;
    ml[kBM + r] = have_o ? l_sum : 0.f;  // l = 0: no visible key, or no tile at all
    tc::fence_before_sync();
    named_bar_sync(1, kWG * 128);
    tc::fence_after_sync();
    const float* ml0 = reinterpret_cast<const float*>(smem + kOffML);
    const float* ml1 = reinterpret_cast<const float*>(smem + kOffML + kTileK);
    const float m0 = ml0[r], l0 = ml0[kBM + r], m1 = ml1[r], l1 = ml1[kBM + r];
    const bool use0 = l0 > 0.f, use1 = l1 > 0.f;
    // the sink logit (arms) is one more term of the denominator, in log2 units
    const bool sink = ARMS && p.sinks != nullptr;
    const float zs = sink ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
    const float M = fmaxf(fmaxf(use0 ? m0 : -INFINITY, use1 ? m1 : -INFINITY), zs);
    const float a0 = use0 ? ex2f((m0 - M) * qs) : 0.f;
    const float a1 = use1 ? ex2f((m1 - M) * qs) : 0.f;
    const float l = a0 * l0 + a1 * l1 + (sink ? ex2f(zs - M) : 0.f);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float c0 = a0 * inv, c1 = a1 * inv;
    // this warpgroup's d_v / 2 of the d_v columns, 32 at a time; O_1 exists once
    // warpgroup 1 had a tile. The output tile goes over Q (every S MMA, the
    // readers of Q, is done), in the 128-byte swizzle of the output's tensor map:
    // column c of row r in block c / 64, 16-byte chunk (c % 64) / 8 XOR r % 8.
    unsigned char* so = smem + kOffOut;
#pragma unroll
    for (int cc = 0; cc < DV / 64; ++cc) {
      const int col0 = wg * (DV / 2) + cc * 32;
      uint32_t o0[32], o1[32];
      tc::tmem_ld_32x32b_x32(tmem + lane_addr + C::col_o(0) + col0, o0);
      if (n_kv > 1) tc::tmem_ld_32x32b_x32(tmem + lane_addr + C::col_o(1) + col0, o1);
      tc::tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        uint32_t w4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = t * 8 + 2 * u;
          float x0 = __uint_as_float(o0[e]) * c0, x1 = __uint_as_float(o0[e + 1]) * c0;
          if (use1) {
            x0 = fmaf(__uint_as_float(o1[e]), c1, x0);
            x1 = fmaf(__uint_as_float(o1[e + 1]), c1, x1);
          }
          w4[u] = pack_bf16(x0, x1);
        }
        const int col = col0 + t * 8;
        const int chunk = (col % 64) / 8;
        *reinterpret_cast<uint4*>(so + (col / 64) * kBlk + r * 128 + ((chunk ^ (r & 7)) * 16)) =
            make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    tc::fence_async_smem();  // the tile visible to the TMA engine
    named_bar_sync(2, kWG * 128);
    if (threadIdx.x == 0) {
      // rows past the end of the sequence fall outside the tensor and are not written
#pragma unroll
      for (int cb = 0; cb < C::kCBV; ++cb) tc::tma_store_4d(&tm_o, so + cb * kBlk, cb * 64, h, i0, b);
      tc::bulk_commit_group();
      tc::bulk_wait_group_read0();  // shared memory stays valid until the store has read it
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kMmaWarp0) tc::tmem_dealloc(tmem, kTmemCols);
}

// A 4-D bf16 tensor of rows of d elements; box = 64 x b1 x b2 x 1 (one 64-column
// block of the rows), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int d, uint64_t d1, uint64_t d2, uint64_t d3, uint32_t box1,
              uint32_t box2) {
  const uint64_t dims[4] = {(uint64_t)d, d1, d2, d3};
  const uint64_t strides[3] = {(uint64_t)d * 2, (uint64_t)d * 2 * d1, (uint64_t)d * 2 * d1 * d2};
  const uint32_t box[4] = {64, box1, box2, 1};
  return make_tmap_bf16(m, base, dims, strides, box);
}

template <int DK, int DV, bool ARMS>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                     const TcParams& p, cudaStream_t st) {
  using C = Cfg<DK, DV>;
  int dev = 0;
  cudaGetDevice(&dev);
  static std::atomic<unsigned long long> attr_done{0};  // per device, per instantiation
  if (dev < 64 && !(attr_done.load(std::memory_order_acquire) >> dev & 1ull)) {
    // The register hand-over inside the kernel assumes exactly kLaunchRegs per
    // thread at launch; with any other allocation it could wait forever, so
    // such a build is refused here instead of launched.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<DK, DV, ARMS>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorNotSupported;
    e = cudaFuncSetAttribute(prefill_tc_kernel<DK, DV, ARMS>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(1ull << dev, std::memory_order_release);
  }
  const long long ctas = (long long)p.B * p.H * p.n_qtiles;
  if (ctas <= 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  // programmatic stream serialization: the CTAs of this launch may start their
  // set-up while the previous kernel in the stream finishes (the kernel waits
  // for it, grid_dep_wait, before touching global memory)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<DK, DV, ARMS>, tq, tk, tv, to, p);
}

}  // namespace

bool prefill_tc_supported(int bf16, int dk, int dv, int bs, int mbps) {
  // (d_k, d_v) = (64, 64), (128, 128) or (192, 128); paged: a pool block is a
  // whole number of 8-row swizzle atoms and divides a 128-key tile, and a table
  // row fits the CTA's shared copy
  const bool widths = (dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 192 && dv == 128);
  return bf16 == 1 && widths &&
         (bs == 0 || (bs % 8 == 0 && kBN % bs == 0 && mbps > 0 && mbps <= kTabEntries));
}

cudaError_t launch_prefill_tc(const void* q, const void* k, const void* v, void* out, int B, int seq_q,
                              int seq_kv_max, const int32_t* offsets, int H, int Hkv, int dk, int dv, float qscale,
                              unsigned* err, cudaStream_t st, const int32_t* tables, int mbps, int bs,
                              int num_blocks, const TcArms* arms, int debug_withhold) {
  if (!prefill_tc_supported(1, dk, dv, tables ? bs : 0, mbps) || !(qscale > 0.f)) return cudaErrorNotSupported;
  CUtensorMap tq, tk, tv, to;
  // q [B, S, H, d_k]: dims (d_k, H, S, B), box (64, 1, 128, 1)
  if (!make_map(&tq, q, dk, H, seq_q, B, 1, kBM)) return cudaErrorInvalidValue;
  if (tables) {
    // pools [num_blocks, Hkv, bs, d]: dims (d, bs, Hkv, num_blocks), box (64, bs, 1, 1)
    if (!make_map(&tk, k, dk, bs, Hkv, num_blocks, bs, 1)) return cudaErrorInvalidValue;
    if (!make_map(&tv, v, dv, bs, Hkv, num_blocks, bs, 1)) return cudaErrorInvalidValue;
  } else {
    // k, v [B, Hkv, S_kv, d]: dims (d, S_kv, Hkv, B), box (64, 128, 1, 1)
    if (!make_map(&tk, k, dk, seq_kv_max, Hkv, B, kBN, 1)) return cudaErrorInvalidValue;
    if (!make_map(&tv, v, dv, seq_kv_max, Hkv, B, kBN, 1)) return cudaErrorInvalidValue;
  }
  // out [B, S, H, d_v]: dims (d_v, H, S, B), box (64, 1, 128, 1)
  if (!make_map(&to, out, dv, H, seq_q, B, 1, kBM)) return cudaErrorInvalidValue;
  TcParams p;
  p.B = B;
  p.S = seq_q;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.S_kv = seq_kv_max;
  p.n_qtiles = (seq_q + kBM - 1) / kBM;
  p.offsets = offsets;
  p.tables = tables;
  p.mbps = mbps;
  p.bs = bs;
  p.num_blocks = num_blocks;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.qscale = qscale;
  p.err = err;
  p.debug_withhold = debug_withhold;
  const bool on = arms && (arms->window > 0 || arms->softcap2 > 0.f || arms->sinks || arms->alibi);
  p.window = on ? arms->window : 0;
  p.cap_out = on ? arms->softcap2 : 0.f;                          // softcap * log2 e
  p.cap_in = on && arms->softcap2 > 0.f ? qscale / arms->softcap2 : 0.f;  // scale / softcap
  p.alibi = on ? arms->alibi : nullptr;
  p.sinks = on ? arms->sinks : nullptr;
  if (on) {
    if (dk == 64) return launch_d<64, 64, true>(tq, tk, tv, to, p, st);
    if (dk == 128) return launch_d<128, 128, true>(tq, tk, tv, to, p, st);
    return launch_d<192, 128, true>(tq, tk, tv, to, p, st);
  }
  if (dk == 64) return launch_d<64, 64, false>(tq, tk, tv, to, p, st);
  if (dk == 128) return launch_d<128, 128, false>(tq, tk, tv, to, p, st);
  return launch_d<192, 128, false>(tq, tk, tv, to, p, st);
}

}  // namespace gqa
