// Instantiations of the SIMT attention kernel for __nv_bfloat16: (d_k, d_v) in (16,16), (32,32), (64,64).
#include "attn_rows.cuh"

namespace gqa {

cudaError_t rows_dispatch_bf16_small(const RowsParams& p, int dk, int dv, int drot, int nv, cudaStream_t st) {
  if (dk == 16 && dv == 16 && drot == 0) {
    if (nv == 1) return launch_rows_inst<__nv_bfloat16, 16, 16, 0, 1>(p, st);
    if (nv == 2) return launch_rows_inst<__nv_bfloat16, 16, 16, 0, 2>(p, st);
  }
  if (dk == 32 && dv == 32 && drot == 0) {
    if (nv == 1) return launch_rows_inst<__nv_bfloat16, 32, 32, 0, 1>(p, st);
    if (nv == 2) return launch_rows_inst<__nv_bfloat16, 32, 32, 0, 2>(p, st);
    if (nv == 4) return launch_rows_inst<__nv_bfloat16, 32, 32, 0, 4>(p, st);
  }
  if (dk == 64 && dv == 64 && drot == 0) {
    if (nv == 1) return launch_rows_inst<__nv_bfloat16, 64, 64, 0, 1>(p, st);
    if (nv == 2) return launch_rows_inst<__nv_bfloat16, 64, 64, 0, 2>(p, st);
    if (nv == 4) return launch_rows_inst<__nv_bfloat16, 64, 64, 0, 4>(p, st);
    if (nv == 8) return launch_rows_inst<__nv_bfloat16, 64, 64, 0, 8>(p, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace gqa
