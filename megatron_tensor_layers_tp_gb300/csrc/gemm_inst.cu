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

template <bool SWAP>
static cudaError_t set_smem_attr() {
  static bool done = false;
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<SWAP, TPK_EPI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e == cudaSuccess) done = true;
  return e;
}

cudaError_t TPK_CAT(launch_gemm_epi, TPK_EPI)(bool swap, const GemmArgs& a, size_t smem,
                                               cudaStream_t st) {
  cudaError_t e = swap ? set_smem_attr<true>() : set_smem_attr<false>();
  if (e != cudaSuccess) return e;
  const int cx = a.cluster_split > 1 ? a.cluster_split : 1;
  if (swap)
    return launch_kc(gemm_kernel<true, TPK_EPI>, dim3(a.grid), dim3(kThreadsOf<true>), smem, st,
                     cx, a);
  return launch_kc(gemm_kernel<false, TPK_EPI>, dim3(a.grid), dim3(kThreadsOf<false>), smem, st,
                   cx, a);
}

// How many clusters of cluster_x CTAs (smem bytes each) can be resident at once.
int TPK_CAT(gemm_max_clusters_epi, TPK_EPI)(bool swap, int cluster_x, size_t smem) {
  if ((swap ? set_smem_attr<true>() : set_smem_attr<false>()) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster_x * 64);
  cfg.blockDim = dim3(swap ? kThreadsOf<true> : kThreadsOf<false>);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e = swap ? cudaOccupancyMaxActiveClusters(&n, gemm_kernel<true, TPK_EPI>, &cfg)
                       : cudaOccupancyMaxActiveClusters(&n, gemm_kernel<false, TPK_EPI>, &cfg);
  return e == cudaSuccess ? n : 0;
}

}  // namespace tpk
