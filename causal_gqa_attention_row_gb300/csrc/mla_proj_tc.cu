// mla_proj_tc.cu -- the per-head projections around the absorbed MLA decode on
// the tcgen05 tensor cores (bf16 inputs, fp32 accumulation): for every head h,
// y[b, h, :M] = W[h] x[b, h, :K] (frink-models src/mla/mod.rs,
// `absorbed_attention`: W = k_b[h] before the attention, v_b[h] after it).
//
// As a product per head, Y_h^T (M x B) = W_h (M x K) X_h^T (K x B): the weight
// rows are the MMA's M (128 per CTA), the batch rows its N (32 per CTA), and
// the K axis is 16 per instruction. One CTA = (128 output rows, head h, 32
// batch rows): the weight tile (128 x K) and the batch rows' slice (32 x K) are
// loaded by TMA in 64-column blocks (128-byte swizzle), one thread issues the
// K / 16 MMAs into a 32-column TMEM accumulator, and the four warps write their
// 32 rows of it (thread = output row m, its 32 columns = the batch rows) to y as
// bf16. Batch rows past B read as zeros and are not written.

#include <atomic>
#include "tc_ptx.cuh"
#include "tmap.h"

namespace gqa {
namespace {

constexpr int kPM = 128, kPN = 32, kPThreads = 128;
constexpr int kMaxKBlocks = 8;  // K <= 512

struct ProjBars {
  uint64_t full, done;
  uint32_t tmem_base;
};

__global__ void __launch_bounds__(kPThreads, 1)
    head_proj_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                        const __nv_bfloat16* __restrict__ x, int x_stride, __nv_bfloat16* __restrict__ y, int y_stride,
                        int B, int H, int M, int K, int tail, unsigned* err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int nkb = K / 64;
  constexpr int kWBlk = kPM * 128, kXBlk = kPN * 128;  // one 64-column block of each tile
  unsigned char* sw = smem;
  unsigned char* sx = smem + nkb * kWBlk;
  ProjBars* bars = reinterpret_cast<ProjBars*>(sx + nkb * kXBlk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kPM, h = blockIdx.y, b0 = blockIdx.z * kPN;
  // launched as a programmatic dependent: x may come from the kernel before this
  // one; the next launch may start setting up at once
  grid_dep_wait();
  grid_dep_launch();

  if (threadIdx.x == 0) {
    mbar_init(&bars->full, 1);
    mbar_init(&bars->done, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&bars->full, nkb * (kWBlk + kXBlk));
    for (int kb = 0; kb < nkb; ++kb) {
      tc::tma_load_4d(sw + kb * kWBlk, &tm_w, kb * 64, m0, h, 0, &bars->full);
      tc::tma_load_4d(sx + kb * kXBlk, &tm_x, kb * 64, h, b0, 0, &bars->full);
    }
  }
  if (warp == 0) {
    tc::tmem_alloc(&bars->tmem_base, 32);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  bool ok = true;
  if (threadIdx.x == 0) {
    ok = mbar_wait(&bars->full, 0);
    if (ok) {
      tc::fence_after_sync();
      const uint32_t idesc = tc::idesc_bf16_f32(kPM, kPN, false);
      constexpr uint64_t kHi = tc::desc_sw128_hi(0, 1024);
      const uint64_t dW = kHi | tc::desc_addr(sw), dX = kHi | tc::desc_addr(sx);
      for (int kk = 0; kk < K / 16; ++kk) {
        const uint32_t aw = (kk / 4) * kWBlk + (kk % 4) * 32, ax = (kk / 4) * kXBlk + (kk % 4) * 32;
        tc::mma_f16_ss(tmem, dW + (aw >> 4), dX + (ax >> 4), idesc, kk > 0);
      }
    } else {
      raise_error(err, kErrTimeout);
    }
    tc::mma_commit(&bars->done);  // also after a timeout: the barrier completes with no MMA
  }
  __syncwarp();
  // every thread: the accumulator is complete (or there is nothing to write)
  ok = mbar_wait(&bars->done, 0) && !(threadIdx.x == 0 && !ok);
  if (!ok && lane == 0) raise_error(err, kErrTimeout);
  tc::fence_after_sync();
  uint32_t d[32];
  tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16), d);
  tc::tmem_ld_wait();
  const int m = m0 + warp * 32 + lane;
  if (m < M) {
#pragma unroll
    for (int j = 0; j < kPN; ++j) {
      const int b = b0 + j;
      if (b < B) y[((size_t)b * H + h) * y_stride + m] = __float2bfloat16_rn(__uint_as_float(d[j]));
    }
  }
  // the columns of x past K are copied to y past M unchanged (the query's rope
  // slice): in 16-byte pieces when the rows allow, every load of a round issued
  // before its stores (one element at a time, each store waited for its load:
  // ~16 round trips per thread)
  if (tail > 0 && blockIdx.x == 0) {
    const bool vec = (tail % 8) == 0 && (x_stride % 8) == 0 && (y_stride % 8) == 0 && (K % 8) == 0 && (M % 8) == 0 &&
                     (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0;
    if (vec) {
      const int per_row = tail / 8, n = kPN * per_row;  // 16-byte pieces
      constexpr int kRound = 4;
      for (int e0 = threadIdx.x; e0 < n; e0 += kRound * kPThreads) {
        uint4 v[kRound];
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
          const int e = e0 + u * kPThreads, b = b0 + e / per_row, c = (e % per_row) * 8;
          if (e < n && b < B) v[u] = *reinterpret_cast<const uint4*>(x + ((size_t)b * H + h) * x_stride + K + c);
        }
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
          const int e = e0 + u * kPThreads, b = b0 + e / per_row, c = (e % per_row) * 8;
          if (e < n && b < B) *reinterpret_cast<uint4*>(y + ((size_t)b * H + h) * y_stride + M + c) = v[u];
        }
      }
    } else {
      for (int e = threadIdx.x; e < kPN * tail; e += kPThreads) {
        const int b = b0 + e / tail, c = e % tail;
        if (b < B) y[((size_t)b * H + h) * y_stride + M + c] = x[((size_t)b * H + h) * x_stride + K + c];
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 32);
}

// A bf16 tensor [d2, d1, d0] with rows of `stride` elements (d0 <= stride);
// box = 64 columns x box1 x box2, 128-byte swizzle, zeros outside.
bool make_map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t stride, uint64_t d1, uint64_t d2,
               uint32_t box1, uint32_t box2) {
  const uint64_t dims[4] = {d0, d1, d2, 1};
  const uint64_t strides[3] = {stride * 2, stride * 2 * d1, stride * 2 * d1 * d2};
  const uint32_t box[4] = {64, box1, box2, 1};
  return make_tmap_bf16(m, base, dims, strides, box);
}

}  // namespace

bool head_proj_tc_supported(int M, int K) { return M % kPM == 0 && K % 64 == 0 && K / 64 <= kMaxKBlocks; }

cudaError_t launch_head_proj_tc(const void* W, const void* x, int x_stride, void* y, int y_stride, int B, int H, int M,
                                int K, int tail, unsigned* err, cudaStream_t st) {
  if (!head_proj_tc_supported(M, K)) return cudaErrorNotSupported;
  if (B == 0) return cudaSuccess;
  CUtensorMap tw, tx;
  // W [H, M, K]: box of 128 rows; x [B, H, x_stride]: box of 1 head x 32 batch rows
  if (!make_map3(&tw, W, (uint64_t)K, (uint64_t)K, (uint64_t)M, (uint64_t)H, kPM, 1)) return cudaErrorInvalidValue;
  if (!make_map3(&tx, x, (uint64_t)K, (uint64_t)x_stride, (uint64_t)H, (uint64_t)B, 1, kPN))
    return cudaErrorInvalidValue;
  const int nkb = K / 64;
  const int smem_bytes = nkb * (kPM + kPN) * 128 + (int)sizeof(ProjBars) + 1024;
  int dev = 0;
  cudaGetDevice(&dev);
  static std::atomic<unsigned long long> attr_done{0};  // per device
  if (dev < 64 && !(attr_done.load(std::memory_order_acquire) >> dev & 1ull)) {
    const cudaError_t e = cudaFuncSetAttribute(head_proj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kMaxKBlocks * (kPM + kPN) * 128 + (int)sizeof(ProjBars) + 1024);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(1ull << dev, std::memory_order_release);
  }
  const dim3 grid((unsigned)(M / kPM), (unsigned)H, (unsigned)((B + kPN - 1) / kPN));
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, head_proj_tc_kernel, tw, tx, static_cast<const __nv_bfloat16*>(x), x_stride,
                            static_cast<__nv_bfloat16*>(y), y_stride, B, H, M, K, tail, err);
}

}  // namespace gqa
