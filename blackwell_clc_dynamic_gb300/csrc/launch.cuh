// Host-side launch helpers for the GEMM kernel instantiations (one translation unit per
// tile / cluster shape so the library builds in parallel).
#pragma once
#include <cuda_runtime.h>

#include "kernel.cuh"

namespace clcg {

// grid_ctas = clusters x CL; the grid is (grid_ctas / CLY) x CLY with clusters of CLX x CLY.
template <int BN, int CL, bool PAIR, int RN = 1>
cudaError_t launch_shape(int sched, const Params& p, int grid_ctas, cudaStream_t stream) {
  using C = Cfg<BN, CL, PAIR, RN>;
  void (*k)(const Params) = nullptr;
  switch (sched) {
    case SCHED_CLC: k = gemm_kernel<BN, CL, PAIR, SCHED_CLC, RN>; break;
    case SCHED_STATIC: k = gemm_kernel<BN, CL, PAIR, SCHED_STATIC, RN>; break;
    case SCHED_NONPERSISTENT: k = gemm_kernel<BN, CL, PAIR, SCHED_NONPERSISTENT, RN>; break;
    default: return cudaErrorInvalidValue;
  }
  if (grid_ctas % CL != 0) return cudaErrorInvalidValue;
  constexpr int smem = C::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid_ctas / C::CLY), C::CLY, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::CLX;
  attr[0].val.clusterDim.y = C::CLY;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, p);
}

// Load the three schedule variants of a shape now and set their shared-memory limit.  With
// CUDA's lazy module loading a kernel's code is loaded at its first launch, and that load
// can wait until the device is idle: a first launch while another kernel holds SMs (an
// occupier spinning on a host flag) would stall until that kernel ends.
template <int BN, int CL, bool PAIR, int RN = 1>
cudaError_t prepare_shape() {
  constexpr int smem = Cfg<BN, CL, PAIR, RN>::SMEM_BYTES;
  void (*ks[3])(const Params) = {gemm_kernel<BN, CL, PAIR, SCHED_CLC, RN>, gemm_kernel<BN, CL, PAIR, SCHED_STATIC, RN>,
                                 gemm_kernel<BN, CL, PAIR, SCHED_NONPERSISTENT, RN>};
  for (auto k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int BN, int CL, bool PAIR, int RN = 1>
cudaError_t max_clusters_shape(int* out) {
  using C = Cfg<BN, CL, PAIR, RN>;
  void (*k)(const Params) = gemm_kernel<BN, CL, PAIR, SCHED_CLC, RN>;
  constexpr int smem = C::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C::CLX * 1024, C::CLY, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::CLX;
  attr[0].val.clusterDim.y = C::CLY;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, (const void*)k, &cfg);
}

// Defined in the per-shape translation units (c2 = CTA pair; c2mc / c4mc = clusters of 2 /
// 4 CTAs with their own MMAs sharing B by multicast; c2x2 = 2 x 2 clusters sharing A along
// rows and B along columns).
cudaError_t launch_n128_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2mc(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c4mc(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2x2(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t max_clusters_n128_c1(int* out);
cudaError_t max_clusters_n256_c1(int* out);
cudaError_t max_clusters_n256_c2(int* out);
cudaError_t max_clusters_n256_c2mc(int* out);
cudaError_t max_clusters_n256_c4mc(int* out);
cudaError_t max_clusters_n256_c2x2(int* out);
cudaError_t prepare_n128_c1();
cudaError_t prepare_n256_c1();
cudaError_t prepare_n256_c2();
cudaError_t prepare_n256_c2mc();
cudaError_t prepare_n256_c4mc();
cudaError_t prepare_n256_c2x2();

// Load every kernel of the library on the current device (see prepare_shape).
inline cudaError_t prepare_all() {
  cudaError_t (*fs[])() = {prepare_n128_c1, prepare_n256_c1, prepare_n256_c2, prepare_n256_c2mc, prepare_n256_c4mc,
                           prepare_n256_c2x2};
  for (auto f : fs) {
    cudaError_t e = f();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The launch function of a shape (nullptr if unsupported).
inline cudaError_t launch_any(int bn, int cl, bool pair, int sched, const Params& p, int grid, cudaStream_t s,
                              int rn = 1) {
  if (cl == 4 && rn == 2) return launch_n256_c2x2(sched, p, grid, s);
  if (cl == 2 && pair) return launch_n256_c2(sched, p, grid, s);
  if (cl == 2) return launch_n256_c2mc(sched, p, grid, s);
  if (cl == 4) return launch_n256_c4mc(sched, p, grid, s);
  if (bn == 128) return launch_n128_c1(sched, p, grid, s);
  return launch_n256_c1(sched, p, grid, s);
}

inline cudaError_t max_clusters_any(int bn, int cl, bool pair, int* out, int rn = 1) {
  if (cl == 4 && rn == 2) return max_clusters_n256_c2x2(out);
  if (cl == 2 && pair) return max_clusters_n256_c2(out);
  if (cl == 2) return max_clusters_n256_c2mc(out);
  if (cl == 4) return max_clusters_n256_c4mc(out);
  if (bn == 128) return max_clusters_n128_c1(out);
  return max_clusters_n256_c1(out);
}

}  // namespace clcg
