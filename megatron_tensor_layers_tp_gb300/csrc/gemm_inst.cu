// One epilogue's instantiations of the sharded tcgen05 GEMM (decode
// orientation with weights on the MMA M side, and prefill orientation with
// tokens on the M side).  Compiled once per epilogue with -DTPK_EPI=<n>.
#include "gemm_kernel.cuh"

#ifndef TPK_EPI
#error "TPK_EPI must be defined"
#endif

namespace tpk {

#define TPK_CAT2(a, b) a##b
#define TPK_CAT(a, b) TPK_CAT2(a, b)

cudaError_t TPK_CAT(launch_gemm_epi, TPK_EPI)(bool swap, const GemmArgs& a, size_t smem,
                                               cudaStream_t st) {
  static bool attr_swap = false, attr_norm = false;
  if (swap) {
    if (!attr_swap) {
      cudaError_t e = cudaFuncSetAttribute(gemm_kernel<true, TPK_EPI>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      attr_swap = true;
    }
    return launch_k(gemm_kernel<true, TPK_EPI>, dim3(a.grid), dim3(kThreads), smem, st, a);
  } else {
    if (!attr_norm) {
      cudaError_t e = cudaFuncSetAttribute(gemm_kernel<false, TPK_EPI>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      attr_norm = true;
    }
    return launch_k(gemm_kernel<false, TPK_EPI>, dim3(a.grid), dim3(kThreads), smem, st, a);
  }
  return cudaGetLastError();
}

}  // namespace tpk
