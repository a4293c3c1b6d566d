// gemm_run_noalloc: the GEMM of gemm_run for callers that cannot allocate device memory.
//
// Some callers can't call cudaMalloc: a process whose device memory is handed entirely
// to its own pool allocator or held under a hard cap, or a latency-critical path where a
// cudaMalloc (which may synchronise the device) is not acceptable.  gemm_run needs a
// handle whose workspace (error word, ownership log) is allocated with cudaMalloc; this
// entry point instead keeps that scratch in one fixed, file-scope device array that
// every GPU which loads the library holds until the process exits.  The caller still
// passes A, B and C.
//
// Limits and sharing:
//   - at most kNoAllocMaxTiles CTA tiles and kNoAllocMaxWorkers launched workers per
//     call; larger problems are rejected with GEMM_ERR_SCRATCH_LIMIT before anything is
//     launched;
//   - every call on a device uses the same array and leaves its contents behind; each
//     call clears the error word on its stream before its kernel and tags its log
//     entries with a per-device launch counter (the array starts zeroed, tag 0 means
//     unwritten, and the log part is cleared again only when the 24-bit tag wraps).
//     Calls that overlap on the GPU (other streams, other threads) race on the array:
//     serialise them.
//   - the first call on a device (with that device current) looks up the array's
//     device address with cudaGetSymbolAddress and launches every kernel once over an
//     empty problem (waiting on a private stream); make that first call before any stream
//     capture begins.
//   - nothing here calls cudaMalloc, cudaFree or an allocating library routine;
//   - gemm_noalloc_status copies the error word and the log of the latest call back to
//     the caller (a wait that ran out leaves C incomplete; that call reports it);
//   - the shapes whose CTAs share operand tiles by TMA multicast run only when the
//     process sees one GPU, and A, B, C must be memory of the current device.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "clcgemm.h"
#include "launch.cuh"

using namespace clcg;

namespace {

constexpr int64_t kNoAllocMaxTiles = 65536;     // CTA tiles (ownership-log entries)
constexpr int64_t kNoAllocMaxWorkers = 65536;   // launched workers (first-tile entries)
constexpr int64_t kErrWords = 4;
constexpr int64_t kScratchWords = kErrWords + 2 * kNoAllocMaxTiles + 2 * kNoAllocMaxWorkers;   // 1 MiB + 16 B

// [0, 4) error word | owner[kNoAllocMaxTiles] | claims[kNoAllocMaxTiles] |
// first[kNoAllocMaxWorkers] (64-bit entries, 8-byte aligned)
static __device__ __align__(256) int32_t g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_dev[kMaxDevices];   // device address of g_noalloc_scratch, per device
int g_sms[kMaxDevices];
bool g_single_gpu[kMaxDevices];        // the process sees one GPU: multicast shapes allowed
uint32_t g_epoch[kMaxDevices];         // log tag of the device's most recent call
int64_t g_last_tiles[kMaxDevices];     // CTA tiles and launched workers of that call (-1: none yet)
int64_t g_last_workers[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return GEMM_OK;
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver || e == cudaErrorInitializationError)
    return GEMM_ERR_NO_DEVICE;
  return GEMM_ERR_CUDA;
}

// Once per device, with that device current: resolve the scratch array's device address.
int setup_device(int dev) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_INVALID_ARG;
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return GEMM_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (g_scratch_dev[dev]) return GEMM_OK;
  int major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
  int n_dev = 0;
  e = cudaGetDeviceCount(&n_dev);
  if (e != cudaSuccess) return from_cuda(e);
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) return from_cuda(e == cudaSuccess ? cudaErrorUnknown : e);
  // launch every kernel this device may run once over an empty problem now, rather than
  // have a first launch load code later (see warm_all); the error words of the scratch
  // take any report
  cudaStream_t st = nullptr;
  e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
  if (e != cudaSuccess) return from_cuda(e);
  e = warm_all(static_cast<int32_t*>(p), st, n_dev == 1);
  cudaStreamDestroy(st);
  if (e != cudaSuccess) return from_cuda(e);
  g_scratch_dev[dev] = static_cast<int32_t*>(p);
  g_sms[dev] = sms;
  g_single_gpu[dev] = n_dev == 1;
  g_last_tiles[dev] = -1;
  g_last_workers[dev] = -1;
  return GEMM_OK;
}

int encode(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
           uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle_bytes) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle swz = swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INVALID_ARG;
}

}  // namespace

extern "C" int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, float* C,
                                gemm_tile_t tile, gemm_cluster_t cluster, gemm_sched_t sched, int num_workers,
                                void* stream) {
  // argument rules of gemm_run
  if (M < 0 || N < 0 || K < 0 || num_workers < 0) return GEMM_ERR_INVALID_ARG;
  if (sched != GEMM_SCHED_CLC && sched != GEMM_SCHED_STATIC && sched != GEMM_SCHED_NONPERSISTENT)
    return GEMM_ERR_INVALID_ARG;
  if (tile.bm != 128 || tile.bk != 64 || cluster.z != 1) return GEMM_ERR_INVALID_ARG;
  int bn = 0, cl = 0, rn = 1;
  bool pair = false;   // clusters of 2 run the CTA-pair MMA (the default options)
  if (cluster.y != 1 && !(cluster.x == 2 && cluster.y == 2)) return GEMM_ERR_INVALID_ARG;
  if (cluster.x == 2 && cluster.y == 2 && tile.bn == 256) {
    bn = 256;
    cl = 4;
    rn = 2;
  } else if (cluster.x == 1 && (tile.bn == 128 || tile.bn == 256)) {
    bn = tile.bn;
    cl = 1;
  } else if ((cluster.x == 2 || cluster.x == 4) && tile.bn == 256) {
    bn = 256;
    cl = cluster.x;
    pair = (cl == 2);
  } else {
    return GEMM_ERR_INVALID_ARG;
  }
  if ((K % 8) != 0 || (N % 8) != 0) return GEMM_ERR_ALIGNMENT;
  if (M > (int64_t)INT32_MAX || N > (int64_t)INT32_MAX || K > (int64_t)INT32_MAX) return GEMM_ERR_TOO_LARGE;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(C) || (K > 0 && (misaligned(A) || misaligned(B)))) return GEMM_ERR_ALIGNMENT;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  int rc = setup_device(dev);
  if (rc) return rc;
  if (uses_tma_multicast(cl, pair) && !g_single_gpu[dev]) return GEMM_ERR_MULTICAST;
  if (!on_device(C, dev) || (K > 0 && (!on_device(A, dev) || !on_device(B, dev)))) return GEMM_ERR_INVALID_ARG;

  const int64_t tile_m = (int64_t)BM * (cl / rn), tile_n = (int64_t)bn * rn;   // cluster tile
  const int64_t mt = (M + tile_m - 1) / tile_m;
  const int64_t nt = (N + tile_n - 1) / tile_n;
  const int64_t total = mt * nt;
  const int64_t n_tiles = total * cl;
  int64_t workers = total;
  if (sched == GEMM_SCHED_STATIC) {
    workers = num_workers > 0 ? num_workers : (g_sms[dev] / cl > 0 ? g_sms[dev] / cl : 1);
  }
  if (n_tiles > kNoAllocMaxTiles || workers > kNoAllocMaxWorkers) return GEMM_ERR_SCRATCH_LIMIT;

  int32_t* err = g_scratch_dev[dev];
  int32_t* owner = err + kErrWords;
  uint32_t* claims = reinterpret_cast<uint32_t*>(owner + kNoAllocMaxTiles);
  unsigned long long* first = reinterpret_cast<unsigned long long*>(claims + kNoAllocMaxTiles);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t epoch;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    epoch = g_epoch[dev] + 1;
    if (epoch >= (1u << 24)) epoch = 1;
    g_epoch[dev] = epoch;
    g_last_tiles[dev] = n_tiles;
    g_last_workers[dev] = workers;
  }
  e = cudaMemsetAsync(err, 0, kErrWords * sizeof(int32_t), s);
  if (e == cudaSuccess && epoch == 1) {
    e = cudaMemsetAsync(claims, 0, (size_t)kNoAllocMaxTiles * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(first, 0, (size_t)kNoAllocMaxWorkers * 8, s);
  }
  if (e != cudaSuccess) return from_cuda(e);

  Params p;
  memset(&p, 0, sizeof p);
  const ShapeInfo si = shape_info(bn, cl, pair, rn);
  if (K > 0) {
    rc = encode(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2,
                (uint32_t)si.bk, (uint32_t)si.a_rows, si.a_swizzle);
    if (rc) return rc;
    rc = encode(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, (uint64_t)N, (uint64_t)K, (uint64_t)N * 2, 64,
                (uint32_t)si.bk, 128);
    if (rc) return rc;
  }
  rc = encode(&p.tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, (uint64_t)N, (uint64_t)M, (uint64_t)N * 4,
              (uint32_t)si.epi_chunk, 32, si.c_swizzle);
  if (rc) return rc;
  p.G = 0;
  p.mt = (int)mt;
  p.nt = (int)nt;
  p.total = (int)total;
  p.k_blocks = (int)((K + si.bk - 1) / si.bk);
  p.raster_group = kDefaultRasterGroup;
  p.log_owner = owner;
  p.log_claims = claims;
  p.log_first = first;
  p.log_epoch = epoch;
  p.trace = nullptr;
  p.err = err;
  p.timeout_ns = 2000000000LL;
  p.inject_fail_after = -1;
  p.n_tiles = n_tiles;
  p.n_workers = workers;

  const int grid = (int)(workers * cl);
  e = launch_any(bn, cl, pair, (int)sched, p, grid, s, rn);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

extern "C" int gemm_noalloc_status(int32_t out3[3], int32_t* owner, int32_t* claims, int32_t* first, int64_t n_tiles,
                                   int64_t n_workers, void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_INVALID_ARG;
  int32_t* err;
  uint32_t epoch;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    err = g_scratch_dev[dev];
    if (!err || g_last_tiles[dev] < 0) return GEMM_ERR_INVALID_ARG;   // no call on this device yet
    if ((owner || claims || first) && (n_tiles != g_last_tiles[dev] || n_workers != g_last_workers[dev]))
      return GEMM_ERR_INVALID_ARG;
    epoch = g_epoch[dev];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every copy is ordered after the call on its stream and waited for at once
  auto copy = [&](void* dst, const void* src, size_t bytes) -> cudaError_t {
    cudaError_t x = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s);
    return x == cudaSuccess ? cudaStreamSynchronize(s) : x;
  };
  int32_t w[3] = {0, 0, 0};
  e = copy(w, err, sizeof w);
  if (e != cudaSuccess) return from_cuda(e);
  if (out3) memcpy(out3, w, sizeof w);
  const int32_t* d_owner = err + kErrWords;
  const uint32_t* d_claims = reinterpret_cast<const uint32_t*>(d_owner + kNoAllocMaxTiles);
  const unsigned long long* d_first = reinterpret_cast<const unsigned long long*>(d_claims + kNoAllocMaxTiles);
  // Copied in chunks through small buffers on the stack: entries carry the tag of the
  // call that wrote them, and only the latest call's count as written.
  constexpr int64_t kChunk = 1024;
  uint32_t raw_c[kChunk];
  unsigned long long raw_f[kChunk];
  if (owner && n_tiles > 0) {
    e = copy(owner, d_owner, (size_t)n_tiles * 4);
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (owner || claims) {
    for (int64_t t0 = 0; t0 < n_tiles; t0 += kChunk) {
      const int64_t n = n_tiles - t0 < kChunk ? n_tiles - t0 : kChunk;
      e = copy(raw_c, d_claims + t0, (size_t)n * 4);
      if (e != cudaSuccess) return from_cuda(e);
      for (int64_t i = 0; i < n; ++i) {
        const int32_t cnt = (raw_c[i] >> 8) == epoch ? (int32_t)(raw_c[i] & 0xFFu) : 0;
        if (claims) claims[t0 + i] = cnt;
        if (owner && cnt == 0) owner[t0 + i] = -1;
      }
    }
  }
  if (first) {
    for (int64_t w0 = 0; w0 < n_workers; w0 += kChunk) {
      const int64_t n = n_workers - w0 < kChunk ? n_workers - w0 : kChunk;
      e = copy(raw_f, d_first + w0, (size_t)n * 8);
      if (e != cudaSuccess) return from_cuda(e);
      for (int64_t i = 0; i < n; ++i)
        first[w0 + i] = (uint32_t)(raw_f[i] >> 32) == epoch ? (int32_t)(uint32_t)raw_f[i] : -1;
    }
  }
  if (w[0] != 0) return (w[0] & ERRB_TIMEOUT) ? GEMM_ERR_TIMEOUT : GEMM_ERR_BOUNDS;
  return GEMM_OK;
}
