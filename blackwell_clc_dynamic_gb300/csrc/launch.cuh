// Host-side launch helpers for the GEMM kernel instantiations (one translation unit per
// tile / cluster shape so the library builds in parallel).
#pragma once
#include <cuda_runtime.h>

#include "kernel.cuh"

namespace clcg {

template <int BN, int CL>
cudaError_t launch_shape(int sched, const Params& p, int grid_ctas, cudaStream_t stream) {
  void (*k)(const Params) = nullptr;
  switch (sched) {
    case SCHED_CLC: k = gemm_kernel<BN, CL, SCHED_CLC>; break;
    case SCHED_STATIC: k = gemm_kernel<BN, CL, SCHED_STATIC>; break;
    case SCHED_NONPERSISTENT: k = gemm_kernel<BN, CL, SCHED_NONPERSISTENT>; break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN, CL>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_ctas, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<BN, CL>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

template <int BN, int CL>
cudaError_t max_clusters_shape(int* out) {
  void (*k)(const Params) = gemm_kernel<BN, CL, SCHED_CLC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN, CL>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * 1024, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<BN, CL>::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, (const void*)k, &cfg);
}

// Defined in the per-shape translation units.
cudaError_t launch_n128_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t max_clusters_n128_c1(int* out);
cudaError_t max_clusters_n256_c1(int* out);
cudaError_t max_clusters_n256_c2(int* out);

}  // namespace clcg
