// mla_proj.cu -- the per-head projections around the absorbed MLA decode
// (frink-models src/mla/mod.rs, `absorbed_attention`): the query's nope slice
// into the latent space through k_b[h] ([d_c, d_nope]) before the attention,
// and each head's weighted latent back to the value width through v_b[h]
// ([d_v, d_c]) after it. Both are, per head h, y[b, h, :M] = W[h] x[b, h, :K]
// over the batch: a [B x K] by [K x M] product per head, done here in fp32 on
// bf16 inputs.
//
// One CTA = (64 outputs m, head h, 32 batch rows b); its 256 threads each own
// 4 outputs x 2 batch rows. The K axis goes through shared memory 64 at a time:
// the W slice transposed to [k][m] (a thread's 4 outputs are one 16-byte read)
// and the x slice as [k][b], both widened to fp32, the next slice's global reads
// in flight during this one's FMAs. K, the row strides and the pointers are
// multiples of 8 elements (16 bytes), which the entry points check.
#include "common.cuh"

namespace gqa {
namespace {

constexpr int kTM = 64, kTB = 32, kTK = 64, kProjThreads = 256;

__global__ void __launch_bounds__(kProjThreads)
    head_matvec_kernel(const __nv_bfloat16* __restrict__ W, const __nv_bfloat16* __restrict__ x, int x_stride,
                       __nv_bfloat16* __restrict__ y, int y_stride, int B, int H, int M, int K, int tail) {
  __shared__ __align__(16) float ws[kTK][kTM];
  __shared__ __align__(16) float xs[kTK][kTB];
  const int m0 = blockIdx.x * kTM, h = blockIdx.y, b0 = blockIdx.z * kTB;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;  // outputs m0 + 4 tx .. +3, rows b0 + 2 ty, +1
  // launched as a programmatic dependent: x may come from the kernel before this
  // one; the next launch may start setting up at once
  grid_dep_wait();
  grid_dep_launch();
  const __nv_bfloat16* Wh = W + (size_t)h * M * K;
  float acc[2][4] = {};
  // K is staged 64 at a time: each thread moves kWTasks 16-byte pieces of W and
  // kXTasks of x per chunk (W[h][m0 + i][kc + 8u ..] -> ws[8u ..][i], x likewise
  // -> xs[8u ..][b]; lanes on consecutive rows, so the eight transposed stores of
  // a piece hit 32 different banks). The next chunk's pieces are read from
  // global memory into registers while this chunk's FMAs run.
  constexpr int kWTasks = kTM * (kTK / 8) / kProjThreads, kXTasks = kTB * (kTK / 8) / kProjThreads;
  static_assert(kWTasks * kProjThreads == kTM * (kTK / 8) && kXTasks * kProjThreads == kTB * (kTK / 8), "tasks");
  uint4 wr[kWTasks], xr[kXTasks];
  auto fetch = [&](int kc) {
#pragma unroll
    for (int q = 0; q < kWTasks; ++q) {
      const int e = threadIdx.x + q * kProjThreads, i = e % kTM, u = e / kTM;
      wr[q] = (m0 + i < M && kc + 8 * u < K) ? *reinterpret_cast<const uint4*>(Wh + (size_t)(m0 + i) * K + kc + 8 * u)
                                             : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < kXTasks; ++q) {
      const int e = threadIdx.x + q * kProjThreads, i = e % kTB, u = e / kTB;
      xr[q] = (b0 + i < B && kc + 8 * u < K)
                  ? *reinterpret_cast<const uint4*>(x + ((size_t)(b0 + i) * H + h) * x_stride + kc + 8 * u)
                  : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  fetch(0);
  for (int kc = 0; kc < K; kc += kTK) {
#pragma unroll
    for (int q = 0; q < kWTasks; ++q) {
      const int e = threadIdx.x + q * kProjThreads, i = e % kTM, u = e / kTM;
      float f[8];
      Elem<__nv_bfloat16>::chunk_to_f32(wr[q], f);
#pragma unroll
      for (int v = 0; v < 8; ++v) ws[8 * u + v][i] = f[v];
    }
#pragma unroll
    for (int q = 0; q < kXTasks; ++q) {
      const int e = threadIdx.x + q * kProjThreads, i = e % kTB, u = e / kTB;
      float f[8];
      Elem<__nv_bfloat16>::chunk_to_f32(xr[q], f);
#pragma unroll
      for (int v = 0; v < 8; ++v) xs[8 * u + v][i] = f[v];
    }
    __syncthreads();
    if (kc + kTK < K) fetch(kc + kTK);
#pragma unroll 8
    for (int j = 0; j < kTK; ++j) {
      const float4 w4 = *reinterpret_cast<const float4*>(&ws[j][4 * tx]);
      const float2 x2 = *reinterpret_cast<const float2*>(&xs[j][2 * ty]);
      acc[0][0] = fmaf(w4.x, x2.x, acc[0][0]);
      acc[0][1] = fmaf(w4.y, x2.x, acc[0][1]);
      acc[0][2] = fmaf(w4.z, x2.x, acc[0][2]);
      acc[0][3] = fmaf(w4.w, x2.x, acc[0][3]);
      acc[1][0] = fmaf(w4.x, x2.y, acc[1][0]);
      acc[1][1] = fmaf(w4.y, x2.y, acc[1][1]);
      acc[1][2] = fmaf(w4.z, x2.y, acc[1][2]);
      acc[1][3] = fmaf(w4.w, x2.y, acc[1][3]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int b = b0 + 2 * ty + u;
    if (b >= B) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int m = m0 + 4 * tx + v;
      if (m < M) y[((size_t)b * H + h) * y_stride + m] = __float2bfloat16_rn(acc[u][v]);
    }
  }
  // the columns of x past K are copied to y past M unchanged (the query's rope slice)
  if (tail > 0 && blockIdx.x == 0) {
    for (int e = threadIdx.x; e < kTB * tail; e += kProjThreads) {
      const int b = b0 + e / tail, c = e % tail;
      if (b < B) y[((size_t)b * H + h) * y_stride + M + c] = x[((size_t)b * H + h) * x_stride + K + c];
    }
  }
}

}  // namespace

cudaError_t launch_head_matvec(const void* W, const void* x, int x_stride, void* y, int y_stride, int B, int H, int M,
                               int K, int tail, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  const dim3 grid((unsigned)((M + kTM - 1) / kTM), (unsigned)H, (unsigned)((B + kTB - 1) / kTB));
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kProjThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, head_matvec_kernel, static_cast<const __nv_bfloat16*>(W),
                            static_cast<const __nv_bfloat16*>(x), x_stride, static_cast<__nv_bfloat16*>(y), y_stride, B,
                            H, M, K, tail);
}

}  // namespace gqa
