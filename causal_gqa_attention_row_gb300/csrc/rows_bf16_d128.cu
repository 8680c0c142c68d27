// Instantiations of the SIMT attention kernel for __nv_bfloat16: (d_k, d_v) in (128,128).
#include "attn_rows.cuh"

namespace gqa {

cudaError_t rows_dispatch_bf16_d128(const RowsParams& p, int dk, int dv, int drot, int nv, cudaStream_t st) {
  if (dk == 128 && dv == 128 && drot == 0) {
    if (nv == 1) return launch_rows_inst<__nv_bfloat16, 128, 128, 0, 1>(p, st);
    if (nv == 2) return launch_rows_inst<__nv_bfloat16, 128, 128, 0, 2>(p, st);
    if (nv == 4) return launch_rows_inst<__nv_bfloat16, 128, 128, 0, 4>(p, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace gqa
