// Instantiations of the SIMT attention kernel for float: (d_k, d_v) in (128,128), (256,256), (192,128), (192,128, rot 64).
#include "attn_rows.cuh"

namespace gqa {

cudaError_t rows_dispatch_f32_large(const RowsParams& p, int dk, int dv, int drot, int nv, cudaStream_t st) {
  if (dk == 128 && dv == 128 && drot == 0) {
    if (nv == 1) return launch_rows_inst<float, 128, 128, 0, 1>(p, st);
    if (nv == 2) return launch_rows_inst<float, 128, 128, 0, 2>(p, st);
    if (nv == 4) return launch_rows_inst<float, 128, 128, 0, 4>(p, st);
  }
  if (dk == 256 && dv == 256 && drot == 0) {
    if (nv == 1) return launch_rows_inst<float, 256, 256, 0, 1>(p, st);
    if (nv == 2) return launch_rows_inst<float, 256, 256, 0, 2>(p, st);
  }
  if (dk == 192 && dv == 128 && drot == 0) {
    if (nv == 1) return launch_rows_inst<float, 192, 128, 0, 1>(p, st);
    if (nv == 2) return launch_rows_inst<float, 192, 128, 0, 2>(p, st);
  }
  if (dk == 192 && dv == 128 && drot == 64) {
    if (nv == 1) return launch_rows_inst<float, 192, 128, 64, 1>(p, st);
    if (nv == 2) return launch_rows_inst<float, 192, 128, 64, 2>(p, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace gqa
