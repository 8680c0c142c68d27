// prefill_tc.cu -- causal prefill on the tcgen05 tensor cores (bf16, d_k = d_v = 64).
//
// The operation (kopitiam-runtime src/attention.rs, `attention_forward` and
// `causal_mask`): row i of sequence b, query head h, sits at position
// offset_b + i and attends to keys 0..=offset_b + i of KV head h / G with
// softmax(scale * q.k); everything else weighs exactly zero.
//
// One CTA = one (sequence, query head, 128-row query tile); CTAs are ordered
// longest-first (the causal work of a tile grows with its index). Roles:
//   warp 0      TMA producer: the Q tile once, then 128-key K and V tiles into a
//               two-stage ring (128-byte swizzle, the layout the MMA reads).
//   warp 1      allocates TMEM; one thread issues every tcgen05.mma:
//               S = Q K^T (M=128, N=128, K=64) into TMEM columns [0,128), and
//               O += P V (M=128, N=64, K=128) into TMEM columns [128,192).
//   warps 2-5   softmax: thread t owns query row t (TMEM lane t). It reads its S
//               row from TMEM, applies the causal mask (only tiles that cross the
//               diagonal), keeps an online softmax with lazy rescaling (O is
//               rescaled in TMEM only when the row maximum grows by more than
//               2^8), writes P as bf16 into shared memory in the swizzled K-major
//               layout, and finally normalises O and stores the output rows.
// S is computed for tile j+1 while the softmax works on tile j.
#include <cudaTypedefs.h>

#include "tc_ptx.cuh"

namespace gqa {
namespace {

constexpr int kD = 64;     // head width (d_k = d_v)
constexpr int kBM = 128;   // query rows per tile
constexpr int kBN = 128;   // keys per tile
constexpr int kStagesKV = 2;
constexpr int kThreads = 192;
constexpr int kTile = kBM * kD * 2;  // 16 KiB: one Q, K or V tile (128 rows x 128 bytes)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColO = 128;
constexpr float kRescaleLog2 = 8.0f;

// shared-memory map (from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffKV = kTile;                              // stage s: K at +0, V at +kTile
constexpr int kOffP = kOffKV + kStagesKV * 2 * kTile;      // P: two 64-key halves
constexpr int kOffBar = kOffP + 2 * kTile;
constexpr int kSmemBytes = kOffBar + 256 + 1024;           // + alignment slack

struct TcParams {
  int B, S, H, Hkv, G, S_kv, n_qtiles;
  const int32_t* offsets;
  __nv_bfloat16* out;
  float qscale;
  unsigned* err;
};

struct Bars {
  uint64_t q_full, kv_full[kStagesKV], kv_empty[kStagesKV], s_full, s_free, p_full, o_done, mma_final;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* bars, unsigned* err) {
  if (*reinterpret_cast<volatile int*>(&bars->abort_flag)) return false;
  if (mbar_wait(bar, parity)) return true;
  *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
  raise_error(err, kErrTimeout);
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item, longest first
  const int per_tile = p.B * p.H;
  const int qt = p.n_qtiles - 1 - (int)(blockIdx.x / per_tile);
  const int rem = (int)(blockIdx.x % per_tile);
  const int h = rem % p.H, b = rem / p.H;
  const int kvh = h / p.G;
  const int i0 = qt * kBM;
  const int off = p.offsets ? p.offsets[b] : 0;
  const int rows = min(kBM, p.S - i0);

  if (off < 0 || (long long)off + p.S > p.S_kv) {  // the cache cannot hold these rows
    if (threadIdx.x == 0 && qt == p.n_qtiles - 1 && h == 0) raise_error(p.err, kErrBounds);
    for (int idx = threadIdx.x; idx < rows * kD; idx += blockDim.x)
      p.out[(((size_t)b * p.S + i0 + idx / kD) * p.H + h) * kD + idx % kD] = __float2bfloat16_rn(0.f);
    return;
  }
  const int n_kv = (off + i0 + rows - 1) / kBN + 1;  // key tiles up to the last row's position

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStagesKV; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 128);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->mma_final, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      tc::prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(&bars->q_full, kTile);
      tc::tma_load_4d(smem + kOffQ, &tm_q, 0, h, i0, b, &bars->q_full);
      int issued_last[kStagesKV] = {-1, -1};
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kStagesKV;
        if (j >= kStagesKV && !wait_or_abort(&bars->kv_empty[st], ((j / kStagesKV) - 1) & 1, bars, p.err)) break;
        mbar_arrive_expect_tx(&bars->kv_full[st], 2 * kTile);
        tc::tma_load_4d(smem + kOffKV + st * 2 * kTile, &tm_k, 0, j * kBN, kvh, b, &bars->kv_full[st]);
        tc::tma_load_4d(smem + kOffKV + st * 2 * kTile + kTile, &tm_v, 0, j * kBN, kvh, b, &bars->kv_full[st]);
        issued_last[st] = j;
      }
      // never exit with a load in flight
      if (!mbar_wait(&bars->q_full, 0)) raise_error(p.err, kErrTimeout);
      for (int st = 0; st < kStagesKV; ++st)
        if (issued_last[st] >= 0 && !mbar_wait(&bars->kv_full[st], (issued_last[st] / kStagesKV) & 1))
          raise_error(p.err, kErrTimeout);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      const uint32_t idS = tc::idesc_bf16_f32(kBM, kBN, false);
      const uint32_t idO = tc::idesc_bf16_f32(kBM, kD, true);
      const uint32_t sQ = smem_u32(smem + kOffQ), sP = smem_u32(smem + kOffP);
      bool ok = wait_or_abort(&bars->q_full, 0, bars, p.err);
      auto issue_s = [&](int j) -> bool {
        const int st = j % kStagesKV;
        if (!wait_or_abort(&bars->kv_full[st], (j / kStagesKV) & 1, bars, p.err)) return false;
        tc::fence_after_sync();
        const uint32_t sK = smem_u32(smem + kOffKV + st * 2 * kTile);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          tc::mma_f16_ss(tmem + kColS, tc::smem_desc_sw128(sQ + kk * 32, 0, 1024),
                         tc::smem_desc_sw128(sK + kk * 32, 0, 1024), idS, kk > 0);
        tc::mma_commit(&bars->s_full);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          ok = wait_or_abort(&bars->s_free, j & 1, bars, p.err) && issue_s(j + 1);
          if (!ok) break;
        }
        if (!wait_or_abort(&bars->p_full, j & 1, bars, p.err)) break;
        tc::fence_after_sync();
        const int st = j % kStagesKV;
        const uint32_t sV = smem_u32(smem + kOffKV + st * 2 * kTile + kTile);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc::mma_f16_ss(tmem + kColO, tc::smem_desc_sw128(sP + (kk / 4) * kTile + (kk % 4) * 32, 0, 1024),
                         tc::smem_desc_sw128(sV + kk * 2048, 0, 1024), idO, (j > 0 || kk > 0));
        tc::mma_commit(&bars->o_done);
        tc::mma_commit(&bars->kv_empty[st]);
      }
      // every MMA issued above has completed before TMEM is released
      tc::mma_commit(&bars->mma_final);
      if (!mbar_wait(&bars->mma_final, 0)) raise_error(p.err, kErrTimeout);
    }
  } else {
    // ================= softmax warps (2..5) =================
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;       // query row within the tile
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int pos = off + i0 + r;            // absolute position of this row
    const float qs = p.qscale;
    const float th = kRescaleLog2 / qs;
    float m_ref = -INFINITY, l = 0.f;
    unsigned char* sP = smem + kOffP;
    bool alive = true;
    for (int j = 0; j < n_kv && alive; ++j) {
      bool ok = mbar_wait(&bars->s_full, j & 1) && !*reinterpret_cast<volatile int*>(&bars->abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
          raise_error(p.err, kErrTimeout);
        }
        alive = false;
        break;
      }
      tc::fence_after_sync();
      float s[kBN];
      {
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          tc::tmem_ld_32x32b_x32(tmem + lane_addr + kColS + c * 32, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(v[e]);
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&bars->s_free);

      const int j0 = j * kBN;
      if (j0 + kBN - 1 > off + i0) {  // this tile crosses the diagonal of some row
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (j0 + c > pos) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kBN; ++c) mx = fmaxf(mx, s[c]);
      float f = 1.f;
      const bool grow = mx > m_ref + th;
      if (grow) {
        f = exp2f((m_ref - mx) * qs);  // 0 while m_ref = -inf
        l *= f;
        m_ref = mx;
      }
      const float mq = m_ref * qs;
      float sum = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        const float p0 = exp2f(fmaf(s[c], qs, -mq));
        const float p1 = exp2f(fmaf(s[c + 1], qs, -mq));
        sum += p0 + p1;
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        pk[c / 2] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      l += sum;

      if (j > 0) {  // PV of tile j-1 done: P may be overwritten and O is stable
        ok = mbar_wait(&bars->o_done, (j - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) raise_error(p.err, kErrTimeout);
          alive = false;
          break;
        }
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, grow)) {  // rescale O in TMEM (rare)
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < kD / 32; ++c) {
            tc::tmem_ld_32x32b_x32(tmem + lane_addr + kColO + c * 32, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tc::tmem_st_32x32b_x32(tmem + lane_addr + kColO + c * 32, o);
          }
          tc::tmem_st_wait();
        }
      }
      // P row r, 128 keys as two 64-key halves, 128-byte swizzle (16-byte chunk
      // index XOR row % 8) -- the K-major layout the PV MMA reads.
#pragma unroll
      for (int cidx = 0; cidx < kBN / 8; ++cidx) {
        const int half = cidx / 8, ch = cidx % 8;
        uint4* dst = reinterpret_cast<uint4*>(sP + half * kTile + r * 128 + ((ch ^ (r & 7)) * 16));
        *dst = make_uint4(pk[cidx * 4], pk[cidx * 4 + 1], pk[cidx * 4 + 2], pk[cidx * 4 + 3]);
      }
      tc::fence_async_smem();
      tc::fence_before_sync();
      mbar_arrive(&bars->p_full);
    }
    // ---- epilogue: O / l -> bf16 rows
    if (alive) {
      const bool ok = mbar_wait(&bars->o_done, (n_kv - 1) & 1);
      if (__all_sync(0xffffffffu, ok)) {
        tc::fence_after_sync();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow = p.out + (((size_t)b * p.S + i0 + r) * p.H + h) * kD;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tc::tmem_ld_32x32b_x32(tmem + lane_addr + kColO + c * 32, o);
          tc::tmem_ld_wait();
          if (r < rows) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(o[e + 2 * t]) * inv,
                                                                __uint_as_float(o[e + 2 * t + 1]) * inv);
                w[t] = *reinterpret_cast<const uint32_t*>(&v2);
              }
              *reinterpret_cast<uint4*>(orow + c * 32 + e) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else if (lane == 0) {
        raise_error(p.err, kErrTimeout);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// A 4-D bf16 tensor of rows of 64 elements; box = 64 x b1 x b2 x 1, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t d1, uint64_t d2, uint64_t d3, uint32_t box1, uint32_t box2) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {kD, d1, d2, d3};
  const cuuint64_t strides[3] = {kD * 2, kD * 2 * d1, kD * 2 * d1 * d2};
  const cuuint32_t box[4] = {kD, box1, box2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(int bf16, int dk, int dv) { return bf16 == 1 && dk == kD && dv == kD; }

cudaError_t launch_prefill_tc(const void* q, const void* k, const void* v, void* out, int B, int seq_q,
                              int seq_kv_max, const int32_t* offsets, int H, int Hkv, int dk, int dv, float qscale,
                              unsigned* err, cudaStream_t st) {
  if (dk != kD || dv != kD || !(qscale > 0.f)) return cudaErrorNotSupported;
  CUtensorMap tq, tk, tv;
  // q [B, S, H, 64]: dims (64, H, S, B), box (64, 1, 128, 1)
  if (!make_map(&tq, q, H, seq_q, B, 1, kBM)) return cudaErrorInvalidValue;
  // k, v [B, Hkv, S_kv, 64]: dims (64, S_kv, Hkv, B), box (64, 128, 1, 1)
  if (!make_map(&tk, k, seq_kv_max, Hkv, B, kBN, 1)) return cudaErrorInvalidValue;
  if (!make_map(&tv, v, seq_kv_max, Hkv, B, kBN, 1)) return cudaErrorInvalidValue;
  TcParams p;
  p.B = B;
  p.S = seq_q;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.S_kv = seq_kv_max;
  p.n_qtiles = (seq_q + kBM - 1) / kBM;
  p.offsets = offsets;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.qscale = qscale;
  p.err = err;
  int dev = 0;
  cudaGetDevice(&dev);
  static unsigned long long attr_done = 0;
  if (dev < 64 && !(attr_done >> dev & 1ull)) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done |= 1ull << dev;
  }
  const long long ctas = (long long)B * H * p.n_qtiles;
  if (ctas <= 0) return cudaSuccess;
  prefill_tc_kernel<<<(unsigned)ctas, kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace gqa
