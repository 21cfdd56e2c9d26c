// One epilogue's instantiations of the sharded tcgen05 GEMM (decode
// orientation with weights on the MMA M side, prefill orientation with tokens
// on the M side, and the prefill orientation on CTA pairs).  Compiled once per
// epilogue with -DTPK_EPI=<n>.
#include "gemm_pair.cuh"

#ifndef TPK_EPI
#error "TPK_EPI must be defined"
#endif

namespace tpk {

#define TPK_CAT2(a, b) a##b
#define TPK_CAT(a, b) TPK_CAT2(a, b)

// the pair kernel serves the epilogues of the prefill orientation
constexpr bool kHasPair = TPK_EPI != EPI_QKV_PIECES;

template <typename F>
static cudaError_t set_smem_attr(F* kernel, bool& done) {
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       227 * 1024);
  if (e == cudaSuccess) done = true;
  return e;
}

static cudaError_t prepare(bool swap, bool pair) {
  static bool done[3] = {false, false, false};
  if (pair) {
    if constexpr (kHasPair) return set_smem_attr(gemm_pair_kernel<TPK_EPI>, done[2]);
    return cudaErrorInvalidValue;
  }
  return swap ? set_smem_attr(gemm_kernel<true, TPK_EPI>, done[1])
              : set_smem_attr(gemm_kernel<false, TPK_EPI>, done[0]);
}

cudaError_t TPK_CAT(launch_gemm_epi, TPK_EPI)(bool swap, const GemmArgs& a, size_t smem,
                                               cudaStream_t st) {
  const bool pair = !swap && a.pair;
  cudaError_t e = prepare(swap, pair);
  if (e != cudaSuccess) return e;
  if (pair) {
    if constexpr (kHasPair)
      return launch_kc(gemm_pair_kernel<TPK_EPI>, dim3(a.grid), dim3(kPairThreads<TPK_EPI>), smem, st,
                       2, a);
    return cudaErrorInvalidValue;
  }
  const int cx = a.cluster_split > 1 ? a.cluster_split : 1;
  if (swap)
    return launch_kc(gemm_kernel<true, TPK_EPI>, dim3(a.grid), dim3(kThreadsOf<true>), smem, st,
                     cx, a);
  return launch_kc(gemm_kernel<false, TPK_EPI>, dim3(a.grid), dim3(kThreadsOf<false>), smem, st,
                   cx, a);
}

// How many clusters of cluster_x CTAs (smem bytes each) can be resident at once.
int TPK_CAT(gemm_max_clusters_epi, TPK_EPI)(bool swap, bool pair, int cluster_x, size_t smem) {
  pair = pair && !swap;
  if (prepare(swap, pair) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster_x * 64);
  cfg.blockDim = dim3(pair ? kPairThreads<TPK_EPI> : (swap ? kThreadsOf<true> : kThreadsOf<false>));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e;
  if (pair) {
    if constexpr (kHasPair) e = cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<TPK_EPI>, &cfg);
    else e = cudaErrorInvalidValue;
  } else {
    e = swap ? cudaOccupancyMaxActiveClusters(&n, gemm_kernel<true, TPK_EPI>, &cfg)
             : cudaOccupancyMaxActiveClusters(&n, gemm_kernel<false, TPK_EPI>, &cfg);
  }
  return e == cudaSuccess ? n : 0;
}

}  // namespace tpk
