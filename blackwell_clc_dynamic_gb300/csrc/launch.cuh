// Host-side launch helpers for the GEMM kernel instantiations (one translation unit per
// tile / cluster shape so the library builds in parallel).
#pragma once
#include <cuda_runtime.h>

#include "kernel.cuh"

namespace clcg {

template <int BN, int CL, bool PAIR>
cudaError_t launch_shape(int sched, const Params& p, int grid_ctas, cudaStream_t stream) {
  void (*k)(const Params) = nullptr;
  switch (sched) {
    case SCHED_CLC: k = gemm_kernel<BN, CL, PAIR, SCHED_CLC>; break;
    case SCHED_STATIC: k = gemm_kernel<BN, CL, PAIR, SCHED_STATIC>; break;
    case SCHED_NONPERSISTENT: k = gemm_kernel<BN, CL, PAIR, SCHED_NONPERSISTENT>; break;
    default: return cudaErrorInvalidValue;
  }
  constexpr int smem = Cfg<BN, CL, PAIR>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_ctas, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, p);
}

template <int BN, int CL, bool PAIR>
cudaError_t max_clusters_shape(int* out) {
  void (*k)(const Params) = gemm_kernel<BN, CL, PAIR, SCHED_CLC>;
  constexpr int smem = Cfg<BN, CL, PAIR>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * 1024, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, (const void*)k, &cfg);
}

// Defined in the per-shape translation units (c2 = CTA pair; c2mc / c4mc = clusters of 2 /
// 4 CTAs with their own MMAs sharing B by multicast).
cudaError_t launch_n128_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2mc(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c4mc(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t max_clusters_n128_c1(int* out);
cudaError_t max_clusters_n256_c1(int* out);
cudaError_t max_clusters_n256_c2(int* out);
cudaError_t max_clusters_n256_c2mc(int* out);
cudaError_t max_clusters_n256_c4mc(int* out);

// The launch function of a shape (nullptr if unsupported).
inline cudaError_t launch_any(int bn, int cl, bool pair, int sched, const Params& p, int grid, cudaStream_t s) {
  if (cl == 2 && pair) return launch_n256_c2(sched, p, grid, s);
  if (cl == 2) return launch_n256_c2mc(sched, p, grid, s);
  if (cl == 4) return launch_n256_c4mc(sched, p, grid, s);
  if (bn == 128) return launch_n128_c1(sched, p, grid, s);
  return launch_n256_c1(sched, p, grid, s);
}

inline cudaError_t max_clusters_any(int bn, int cl, bool pair, int* out) {
  if (cl == 2 && pair) return max_clusters_n256_c2(out);
  if (cl == 2) return max_clusters_n256_c2mc(out);
  if (cl == 4) return max_clusters_n256_c4mc(out);
  if (bn == 128) return max_clusters_n128_c1(out);
  return max_clusters_n256_c1(out);
}

}  // namespace clcg
