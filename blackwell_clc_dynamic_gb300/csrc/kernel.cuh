// Warp-specialised, output-tile-scheduled bf16 GEMM for sm_103a (C = A * B, fp32 out).
//
// One CTA (or CTA pair) computes one output tile at a time:
//   warp 0      TMA producer: A[128 x BK] and B[BK x BN] k-slices (BK = 32 or 64) into a
//               swizzled ring; in multicast clusters each CTA loads its share of the tiles
//               its cluster row / column shares and multicasts it
//   warp 1      MMA issuer (every CTA; only rank 0 of a CTA pair): tcgen05.mma kind::f16
//               into a double-buffered TMEM accumulator; also allocates / frees tensor memory
//   warp 2      CLC scheduler (CTA rank 0, CLC mode only): try_cancel into a 3-deep ring of
//               16-byte responses, bounded by a throttle pipeline
//   warp 3      spare
//   warps 4..7  epilogue: TMEM -> registers -> swizzled shared memory -> TMA store of fp32 C
//               (a CTA's last tile is staged whole in the idle operand ring, without
//               waiting for one store to release a buffer before the next)
//
// The schedule (what the "CUTLASS CLC dynamic persistent kernel" page calls the three kinds
// of kernel, section "From one tile per block to one worker working continuously"):
//   SCHED_CLC            grid over all tiles; first tile = own launch coordinate (the ClcID),
//                        later tiles = launches cancelled with clusterlaunchcontrol.try_cancel
//   SCHED_STATIC         grid over W workers; worker w walks tiles w, w+W, w+2W, ...
//   SCHED_NONPERSISTENT  grid over all tiles; each CTA computes its own tile and exits
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "ptx.cuh"

namespace clcg {

enum : int { SCHED_CLC = 0, SCHED_STATIC = 1, SCHED_NONPERSISTENT = 2 };

constexpr int BM = 128;          // rows of C per CTA
constexpr int UMMA_K = 16;       // k per tcgen05.mma kind::f16
constexpr int NUM_THREADS = 256;
constexpr int CLC_DEPTH = 3;     // response ring depth
constexpr int THR_DEPTH = 3;     // throttle ring depth
constexpr int EPI_WARP0 = 4;
constexpr int TRACE_WORDS = 8;   // u64 per CTA tile in the optional trace
// Default raster band height in tile rows.  Against 8-row bands, 16-row bands let the
// tiles running at one time span half as many B columns, so B streams from DRAM half as
// often; the work per SM clock is the same, but under the 1.4 kW power cap the SMs clock
// higher (square 8192^3: +3-8 %; pair, grouped and tail shapes equal or slightly faster).
constexpr int kDefaultRasterGroup = 16;

// Device error word: [0] bits, [1] first failing wait site (or 100 + failed bounds check),
// [2] block of that failure.
enum : int { ERRB_TIMEOUT = 1, ERRB_BOUNDS = 2 };
// Bounds checks of the checked build (compiled with CLCG_BOUNDS_CHECK): which invariant of
// a work tile failed.
#ifdef CLCG_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif
enum : int { CHK_GROUP = 101, CHK_ROW = 102, CHK_COL = 103, CHK_POS = 104, CHK_WORKER = 105, CHK_KB = 106 };
enum : int {
  WAIT_EMPTY = 1, WAIT_FULL = 2, WAIT_ACC_EMPTY = 3, WAIT_ACC_FULL = 4, WAIT_CLC_FULL = 5,
  WAIT_CLC_EMPTY = 6, WAIT_THR_FULL = 7, WAIT_THR_EMPTY = 8
};

struct Params {
  CUtensorMap tmA;               // A: bf16 M x K row-major, box BK(k) x A_OWN_ROWS, swizzle = BK * 2 bytes
  CUtensorMap tmB;               // B: bf16 K x N row-major, box 64(n) x BK(k), 128B swizzle
  CUtensorMap tmC;               // C: fp32 M x N row-major, box EPI_CHUNK x 32, swizzle = EPI_CHUNK * 4 bytes
  const CUtensorMap* gmaps;      // grouped: (A, B, C) per problem in device memory
  const int* g_tile_start;       // grouped: G+1 prefix sums of cluster tiles
  const int* g_mt;               // grouped: cluster-tile rows of each problem
  const int* g_nt;               // grouped: cluster-tile columns of each problem
  const int* g_kb;               // grouped: k-blocks (ceil(K_g / BK)) of each problem
  int G;                         // number of problems (0: plain problem in tmA/tmB/tmC)
  int mt, nt;                    // cluster-tile grid of the plain problem
  int total;                     // cluster tiles in the launch
  int k_blocks;                  // ceil(K / BK)
  int raster_group;              // tile rows per raster band
  // Ownership log.  Entries carry the tag of the launch that wrote them, so a launch needs
  // no clearing pass: an entry with another launch's tag reads as "not written".
  int* log_owner;                // [CTA tiles] worker that computed the tile (or null: no log)
  unsigned* log_claims;          // [CTA tiles] (tag << 8) | times the tile was computed (saturates at 255)
  unsigned long long* log_first; // [launched workers] (tag << 32) | linear id of the worker's first tile
  unsigned log_epoch;            // this launch's tag, in [1, 2^24)
  unsigned long long* trace;     // [CTA tiles][8]: start ns, end ns, smid, worker, producer's wait
                                 // for this tile's CLC response (ns), try_cancel round trip (ns),
                                 // epilogue start ns, last MMA issued ns
  int* err;                      // device error word
  long long timeout_ns;          // bound on every wait
  int inject_fail_after;         // CLC: stop after this many successful cancels (<0: off)
  int l2_prefetch;               // k-blocks the producer prefetches into L2 ahead of its loads (0: off)
  int hold_scheduler;            // test hook: the CLC scheduler issues and signals nothing
  int pdl;                       // launched as a programmatic dependent of the previous kernel
  int fetch_ahead;               // extra throttle tokens: the scheduler fetches this many more tiles ahead
  long long n_tiles;             // CTA tiles of the launch (ownership-log entries); checked build only
  long long n_workers;           // launched workers (first-tile entries); checked build only
};

// Cluster shapes:
//   CL == 1            one CTA, one 128 x BN tile
//   CL == 2, PAIR      a CTA pair runs one tcgen05 cta_group::2 MMA of 256 x BN; each CTA
//                      loads its own 128 rows of A and its own BN/2 columns of B
//   CL == 2 or 4, !PAIR  CL CTAs each run their own 128 x BN MMA on consecutive row blocks
//                      and share the B tile: each loads 1/CL of it and multicasts that part
//                      to every CTA of the cluster
//   CL == 4, RN == 2   a 2 x 2 cluster: each CTA runs its own 128 x BN MMA on one quarter of a
//                      256 x 2BN cluster tile; the two CTAs of a row share their A tile (each
//                      loads half of its rows), the two CTAs of a column share their B tile
//                      (each loads half of its boxes), both by multicast
// RN is the number of CTAs of a cluster along N; RM = CL / RN along M.  Cluster rank r sits
// at row r / RN, column r % RN of the cluster tile.  Clusters with RN == 1 are launched as
// CL x 1 x 1, the 2 x 2 cluster as 2 x 2 x 1 over a (2 * tiles) x 2 grid.
template <int BN_, int CL_, bool PAIR_, int RN_ = 1>
struct Cfg {
  static constexpr int BN = BN_;                // columns of C per CTA tile (MMA N)
  static constexpr int CL = CL_;                // CTAs per cluster
  static constexpr bool PAIR = PAIR_;
  static constexpr int RN = RN_;                // CTAs along N
  static constexpr int RM = CL / RN;            // CTAs along M
  static constexpr int CLX = (RN == 1) ? CL : RN;   // launch cluster dimensions
  static constexpr int CLY = CL / CLX;
  static constexpr bool MCAST = (CL > 1 && !PAIR);
  static constexpr bool A_MCAST = MCAST && RN > 1;   // A shared along a cluster row
  static constexpr int CG = PAIR ? 2 : 1;       // tcgen05 cta_group
  static constexpr int BN_CTA = PAIR ? BN / 2 : BN;   // B columns each CTA holds in shared memory
  static constexpr int MMA_M = PAIR ? 2 * BM : BM;
  // The 128 x 256 per-CTA MMA needs the most operand bytes per MMA cycle; it takes 32-deep
  // k-slices so that nine 24 KiB stages (instead of four of 48 KiB) keep more bytes in
  // flight.  The other shapes take 64-deep slices (128-byte rows of A).
  static constexpr bool FINE = (!PAIR && BN == 256);
  static constexpr int BK = FINE ? 32 : 64;     // k per ring stage
  static constexpr int A_ROW = BK * 2;          // bytes per A row in a stage (64 or 128)
  static constexpr int A_SWZ = FINE ? 4 : 2;    // smem descriptor swizzle code: 4 = 64 B, 2 = 128 B
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN_CTA * BK * 2;
  static constexpr int B_BOXES = BN_CTA / 64;   // 64-column TMA boxes per stage
  static constexpr int B_OWN_BOXES = MCAST ? B_BOXES / RM : B_BOXES;   // B boxes this CTA loads
  static constexpr int A_OWN_ROWS = A_MCAST ? BM / RN : BM;            // A rows this CTA loads
  static constexpr int STAGES = FINE ? 9 : 6;
  // transaction bytes on the full barrier the MMA waits on: the pair's leader counts both
  // CTAs' loads; a multicast CTA receives its A and the whole B tile
  static constexpr int TX_BYTES = PAIR ? (A_BYTES + B_BYTES) * 2 : (A_BYTES + B_BYTES);
  static constexpr int EMPTY_ARRIVALS = MCAST ? CL : 1;   // MMA commits that free a stage
  static constexpr int TMEM_COLS = 2 * BN;      // two accumulators of BN fp32 columns
  static constexpr int EPI_CHUNK = FINE ? 16 : 32;             // fp32 columns per epilogue store
  static constexpr int C_ROW = EPI_CHUNK * 4;                  // bytes per staged C row (64 or 128)
  static constexpr int C_BUFS = FINE ? 1 : 2;                  // staging buffers per epilogue warp
  static constexpr int C_BUF_BYTES = 32 * C_ROW;
  // A CTA's last tile: the operand ring is idle, so each epilogue warp stages its whole 32
  // rows there (one buffer per chunk).  Not in the multicast clusters, whose rings peer
  // CTAs also write.
  static constexpr bool RING_STAGING = !MCAST;
  static constexpr int CHUNKS = BN / EPI_CHUNK;                // stores per epilogue warp per tile
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_C = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_C + 4 * C_BUFS * C_BUF_BYTES;
  // barrier indices
  static constexpr int BAR_FULL = 0, BAR_EMPTY = STAGES, BAR_ACC_FULL = 2 * STAGES,
                       BAR_ACC_EMPTY = 2 * STAGES + 2, BAR_CLC_FULL = 2 * STAGES + 4,
                       BAR_CLC_EMPTY = BAR_CLC_FULL + CLC_DEPTH, BAR_THR_FULL = BAR_CLC_EMPTY + CLC_DEPTH,
                       BAR_THR_EMPTY = BAR_THR_FULL + THR_DEPTH, NUM_BARS = BAR_THR_EMPTY + THR_DEPTH;
  static constexpr int OFF_RESP = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;
  static constexpr int OFF_MISC = OFF_RESP + CLC_DEPTH * 16;   // [0] tmem base [1] abort [2..4] injected
  static constexpr int SMEM_USED = OFF_MISC + 32;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;         // slack to align the base to 1 KiB
  // consumer warps of a CLC response: TMA + 4 epilogue warps in every CTA, the MMA warp of
  // every CTA that issues MMAs, and the scheduler warp of rank 0
  static constexpr int CLC_CONSUMERS = 5 * CL + (PAIR ? 1 : CL) + 1;
  static_assert(!PAIR || (CL == 2 && RN == 1), "CTA pairs only");
  static_assert(CL % RN == 0 && (RN == 1 || (RN == 2 && CL == 4)), "cluster shape");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(BN % EPI_CHUNK == 0 && BN_CTA % 64 == 0 && BK % UMMA_K == 0, "tile shape");
  static_assert(B_BOXES % (MCAST ? RM : 1) == 0, "B boxes split evenly over a cluster column");
  static_assert((A_OWN_ROWS * A_ROW) % 1024 == 0, "A halves start on a swizzle atom");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && C_BUF_BYTES % 1024 == 0, "1 KiB alignment");
  static_assert(!RING_STAGING || 4 * CHUNKS * C_BUF_BYTES <= STAGES * (A_BYTES + B_BYTES), "last tile fits the ring");
};

// Host view of a shape's TMA boxes and k-slice depth.
struct ShapeInfo {
  int bk;          // k per stage (A box width, B box height)
  int a_rows;      // A box height (rows of A one CTA loads per stage)
  int epi_chunk;   // C box width (fp32 columns)
  int a_swizzle;   // bytes: 64 or 128
  int c_swizzle;   // bytes: 64 or 128
  int smem;
};

template <int BN, int CL, bool PAIR, int RN = 1>
constexpr ShapeInfo shape_info_of() {
  using C = Cfg<BN, CL, PAIR, RN>;
  return ShapeInfo{C::BK, C::A_OWN_ROWS, C::EPI_CHUNK, C::A_ROW, C::C_ROW, C::SMEM_BYTES};
}

inline ShapeInfo shape_info(int bn, int cl, bool pair, int rn = 1) {
  if (cl == 4 && rn == 2) return shape_info_of<256, 4, false, 2>();
  if (cl == 2 && pair) return shape_info_of<256, 2, true>();
  if (cl == 2) return shape_info_of<256, 2, false>();
  if (cl == 4) return shape_info_of<256, 4, false>();
  return bn == 128 ? shape_info_of<128, 1, false>() : shape_info_of<256, 1, false>();
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05): start >> 4 in [0,14), leading byte offset >> 4
// in [16,30), stride byte offset >> 4 in [32,46), fixed 0b001 in [46,49), base offset 0,
// swizzle mode in [61,64): 2 = 128-byte swizzle, 4 = 64-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)swz << 61);
}

// A tile, K-major: rows of BK bf16 (A_ROW bytes), 8-row swizzle atoms 8 * A_ROW bytes apart.
template <class C>
__device__ __forceinline__ uint64_t desc_a(uint32_t addr) { return smem_desc(addr, 16, 8 * C::A_ROW, C::A_SWZ); }

// B tile, MN-major: 64-column (128 B) atoms of BK k-rows (BK * 128 B apart along n), 8
// k-rows per 128-byte swizzle atom (1024 B apart along k).
template <class C>
__device__ __forceinline__ uint64_t desc_b(uint32_t addr) { return smem_desc(addr, C::BK * 128, 1024, 2); }

// Instruction descriptor, kind::f16: D f32 (bit 4), A bf16 (bits 7-9 = 1), B bf16 (bits 10-12
// = 1), A K-major (bit 15 = 0), B MN-major (bit 16 = 1), N >> 3 at bit 17, M >> 4 at bit 24.
template <int M, int N>
__device__ __forceinline__ constexpr uint32_t make_idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- tile map
struct Work {
  int c;       // linear cluster-tile id (= launch coordinate of the cluster it came from)
  int g;       // problem
  int m_blk;   // this CTA's 128-row block inside its problem
  int n_blk;   // BN-column block
  int pos;     // ownership-log index of this CTA's tile
  int kb;      // k-blocks of this tile's problem
  bool valid;
  bool skip;   // checked build: a bounds check failed; every role passes over the tile
};

// Checked build: record a failed bounds check in the error word (first failure's site and
// block), never trap.
__device__ __forceinline__ void report_bounds(const Params& p, int site) {
  if ((atomicOr(p.err, ERRB_BOUNDS) & (ERRB_TIMEOUT | ERRB_BOUNDS)) == 0) {
    p.err[1] = site;
    p.err[2] = (int)blockIdx.x;
  }
}

// Raster / swizzle: bands of `group` tile rows; inside a band the row index runs fastest.
__device__ __forceinline__ void raster_map(int c, int mt, int nt, int group, int& m, int& n) {
  const int band = c / (group * nt);
  const int rows = min(group, mt - band * group);
  const int r = c - band * group * nt;
  m = band * group + r % rows;
  n = r / rows;
}

template <int CL, int RN>
__device__ __forceinline__ Work make_work(const Params& p, int c, uint32_t rank) {
  Work w;
  w.c = c;
  w.valid = (c >= 0) && (c < p.total);
  w.g = 0;
  w.m_blk = 0;
  w.n_blk = 0;
  w.pos = 0;
  w.kb = 0;
  w.skip = false;
  if (!w.valid) return w;
  int base = 0, mt = p.mt, nt = p.nt, kb = p.k_blocks, g = 0;
  if (p.G > 0) {
    int lo = 0, hi = p.G - 1;   // largest g with start[g] <= c
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.g_tile_start + mid) <= c) lo = mid; else hi = mid - 1;
    }
    g = lo;
    base = __ldg(p.g_tile_start + g);
    mt = __ldg(p.g_mt + g);
    nt = __ldg(p.g_nt + g);
    kb = __ldg(p.g_kb + g);
  }
  int m, n;
  raster_map(c - base, mt, nt, p.raster_group, m, n);
  w.g = g;
  // rank r: row r / RN, column r % RN of the cluster tile; CTA tiles are numbered row-major
  // over the problem's (mt * RM) x (nt * RN) grid, problems one after another
  w.m_blk = m * (CL / RN) + (int)rank / RN;
  w.n_blk = n * RN + (int)rank % RN;
  w.pos = base * CL + w.m_blk * (nt * RN) + w.n_blk;
  w.kb = kb;
  if constexpr (kBoundsCheck) {
    // Every index the roles derive from the tile: its problem, its row and column block
    // inside the problem's cluster-tile grid, its log entry, its k-loop length.  A failure
    // is recorded and every role passes over the tile (all roles derive the same Work).
    int site = 0;
    if (p.G > 0 && (g < 0 || g >= p.G)) site = CHK_GROUP;
    else if (w.m_blk < 0 || w.m_blk >= mt * (CL / RN)) site = CHK_ROW;
    else if (w.n_blk < 0 || w.n_blk >= nt * RN) site = CHK_COL;
    else if (w.pos < 0 || (long long)w.pos >= p.n_tiles) site = CHK_POS;
    else if (kb < 0) site = CHK_KB;
    if (site) {
      report_bounds(p, site);
      w.skip = true;
    }
  }
  return w;
}

// ---------------------------------------------------------------- ownership log
// Count one more computation of a tile in this launch.  A claim word written by another
// launch (another tag) restarts at 1.  Each failed compare-and-swap means another claimant
// of the same tile succeeded, so the loop ends after at most as many rounds as there are
// claimants; the bound only guards a word that something else keeps rewriting.
__device__ __forceinline__ void log_claim(unsigned* word, unsigned epoch) {
  unsigned old = *reinterpret_cast<volatile unsigned*>(word);
  for (int i = 0; i < 1024; ++i) {
    const unsigned cnt = (old >> 8) == epoch ? min((old & 0xFFu) + 1u, 0xFFu) : 1u;
    const unsigned prev = atomicCAS(word, old, (epoch << 8) | cnt);
    if (prev == old) return;
    old = prev;
  }
}

// ---------------------------------------------------------------- bounded waits
struct Ctl {
  volatile uint32_t* abort;   // shared: set once any wait of this CTA gave up
};

static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, bool cluster_scope, const Params& p,
                                       Ctl ctl, int where) {
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i) {
      const bool ok = cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
      if (ok) return true;
    }
    if (*ctl.abort) return false;
    if ((long long)(globaltimer() - t0) > p.timeout_ns) {
      if (atomicOr(p.err, ERRB_TIMEOUT) == 0) {
        p.err[1] = where;
        p.err[2] = (int)blockIdx.x;
      }
      *ctl.abort = 1;
      return false;
    }
  }
}

template <bool CS = false>
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, const Params& p, Ctl ctl, int where) {
  const bool ok = CS ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  if (ok) return true;
  return wait_slow(bar, parity, CS, p, ctl, where);
}

// ---------------------------------------------------------------- work iterator
// Every role walks the same tile sequence.  In CLC mode each role consumes every response
// of the ring (one release per consuming warp).
template <int BN, int CL, bool PAIR, int SCHED, int RN>
struct WorkIter {
  using C = Cfg<BN, CL, PAIR, RN>;
  int c = 0;
  int stage = 0;
  uint32_t phase = 0;

  __device__ __forceinline__ Work first(const Params& p, uint32_t rank) {
    c = (int)(blockIdx.x / C::CLX);
    return make_work<CL, RN>(p, c, rank);
  }

  // `warp_wide`: all 32 lanes call (one release per warp); otherwise a single lane calls.
  __device__ __forceinline__ Work next(const Params& p, uint32_t rank, uint32_t smem_base, Ctl ctl,
                                       bool warp_wide) {
    if constexpr (SCHED == SCHED_STATIC) {
      c += (int)(gridDim.x / C::CLX);
      return make_work<CL, RN>(p, c, rank);
    } else if constexpr (SCHED == SCHED_NONPERSISTENT) {
      Work w = make_work<CL, RN>(p, -1, rank);
      return w;
    } else {
      const uint32_t full = smem_base + C::OFF_BAR + 8 * (C::BAR_CLC_FULL + stage);
      const uint32_t empty = smem_base + C::OFF_BAR + 8 * (C::BAR_CLC_EMPTY + stage);
      const uint32_t resp = smem_base + C::OFF_RESP + 16 * stage;
      volatile uint32_t* injected = reinterpret_cast<volatile uint32_t*>(
          __cvta_shared_to_generic(smem_base + C::OFF_MISC + 8 + 4 * stage));
      Work w = make_work<CL, RN>(p, -1, rank);
      const bool got = bar_wait<(CL > 1)>(full, phase, p, ctl, WAIT_CLC_FULL);
      if (got) {
        uint32_t x = 0;
        bool ok = false;
        if (*injected == 0) ok = clc_decode(resp, x);   // success predicate first
        fence_proxy_async_smem();                        // reads done before the slot is rewritten
        if (ok) w = make_work<CL, RN>(p, (int)(x / C::CLX), rank);
      }
      if (warp_wide) __syncwarp();
      if (!warp_wide || lane_id() == 0) {
        if (CL == 1 || rank == 0) mbar_arrive(empty);
        else mbar_arrive_cluster(map_to_rank(empty, 0));
      }
      if (++stage == CLC_DEPTH) { stage = 0; phase ^= 1; }
      return w;
    }
  }
};

// ---------------------------------------------------------------- the kernel
template <int BN, int CL, bool PAIR, int SCHED, int RN = 1>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const __grid_constant__ Params p) {
  using C = Cfg<BN, CL, PAIR, RN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = (CL == 1) ? 0u : cluster_ctarank();
  const int worker = (int)(blockIdx.x / C::CLX);   // the cluster's launch id

  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * (uint32_t)i; };
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  Ctl ctl{misc + 1};

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::BAR_FULL + s), 1);
      mbar_init(bar(C::BAR_EMPTY + s), C::EMPTY_ARRIVALS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(C::BAR_ACC_FULL + a), 1);
      mbar_init(bar(C::BAR_ACC_EMPTY + a), PAIR ? 8 : 4);
    }
    for (int i = 0; i < CLC_DEPTH; ++i) {
      mbar_init(bar(C::BAR_CLC_FULL + i), 1);
      mbar_init(bar(C::BAR_CLC_EMPTY + i), C::CLC_CONSUMERS);
    }
    for (int i = 0; i < THR_DEPTH; ++i) {
      mbar_init(bar(C::BAR_THR_FULL + i), 1);
      mbar_init(bar(C::BAR_THR_EMPTY + i), 1);
    }
    for (int i = 1; i < 8; ++i) misc[i] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0 && p.G == 0 && p.k_blocks > 0) {
    prefetch_tmap(&p.tmA);
    prefetch_tmap(&p.tmB);
    prefetch_tmap(&p.tmC);
  }
  if (warp == 1) {
    tmem_alloc<C::CG>(smem_addr((const void*)(smem + C::OFF_MISC)), C::TMEM_COLS);
    tmem_relinquish<C::CG>();
  }
  tc_fence_before();
  if constexpr (CL > 1) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  if (p.pdl) {
    // Programmatic dependent launch: the prologue above touched no global memory, so it may
    // overlap the previous kernel; everything below waits until that kernel has completed
    // and its writes are visible.  The next kernel may be scheduled from now on (it waits
    // the same way before touching memory).
    griddep_launch_dependents();
    griddep_wait();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      WorkIter<BN, CL, PAIR, SCHED, RN> it;
      Work w = it.first(p, rank);
      int s = 0;
      uint32_t ph = 0;
      int tile = 0;
      const uint32_t full0_leader = PAIR ? map_to_rank(bar(C::BAR_FULL), 0) : bar(C::BAR_FULL);
      const int rm = (int)rank / RN, rn = (int)rank % RN;   // place in the cluster tile
      uint16_t col_ctas = 0;   // the CTAs of this cluster column share the B tile
#pragma unroll
      for (int r = 0; r < C::RM; ++r) col_ctas |= (uint16_t)(1u << (r * RN + rn));
      // the CTAs of this cluster row share the A tile (2 x 2 clusters)
      const uint16_t row_ctas = (uint16_t)(((1u << RN) - 1u) << (rm * RN));
      // throttle: one token per tile started; the scheduler issues fetch r only after token
      // r, so it fetches tile r + 1 once tile r - fetch_ahead has started (default: once tile
      // r has started, one tile ahead)
      auto produce_token = [&](int tok) -> bool {
        const int t = tok % THR_DEPTH;
        if (!bar_wait(bar(C::BAR_THR_EMPTY + t), ((tok / THR_DEPTH) & 1) ^ 1, p, ctl, WAIT_THR_EMPTY)) return false;
        mbar_arrive(bar(C::BAR_THR_FULL + t));
        return true;
      };
      const int ahead = (SCHED == SCHED_CLC && rank == 0) ? min(max(p.fetch_ahead, 0), THR_DEPTH - 1) : 0;
      bool tok_ok = true;
      for (int tok = 0; tok < ahead && w.valid && tok_ok; ++tok) tok_ok = produce_token(tok);
      while (w.valid && tok_ok) {
        if (SCHED == SCHED_CLC && rank == 0) {
          if (!produce_token(tile + ahead)) break;
        }
        if (kBoundsCheck && w.skip) {   // checked build: a tile that failed a bounds check
          ++tile;
          w = it.next(p, rank, sb, ctl, false);
          continue;
        }
        if (p.trace) p.trace[TRACE_WORDS * (size_t)w.pos + 0] = globaltimer();
        const CUtensorMap* mA = p.G ? p.gmaps + 3 * w.g : &p.tmA;
        const CUtensorMap* mB = p.G ? p.gmaps + 3 * w.g + 1 : &p.tmB;
        const int ay = w.m_blk * BM;
        const int a_row0 = ay + (C::A_MCAST ? rn * C::A_OWN_ROWS : 0);   // first A row this CTA loads
        const int bx = w.n_blk * BN + (PAIR ? (int)rank * C::BN_CTA : 0);
        const int pf = p.l2_prefetch;
        auto prefetch = [&](int kq) {
          tma_prefetch_l2_2d(mA, kq * C::BK, a_row0);
#pragma unroll
          for (int j = 0; j < C::B_BOXES; ++j) tma_prefetch_l2_2d(mB, bx + 64 * j, kq * C::BK);
        };
        for (int kq = C::STAGES; kq < pf && kq < w.kb; ++kq) prefetch(kq);
        bool ok = true;
        for (int kb = 0; kb < w.kb; ++kb) {
          if (pf > 0 && kb + pf < w.kb && kb + pf >= C::STAGES) prefetch(kb + pf);
          if (!bar_wait<(CL > 1)>(bar(C::BAR_EMPTY + s), ph ^ 1, p, ctl, WAIT_EMPTY)) { ok = false; break; }
          if (!PAIR || rank == 0) mbar_arrive_expect_tx(bar(C::BAR_FULL + s), C::TX_BYTES);
          const uint32_t a_dst = sb + C::OFF_A + (uint32_t)s * C::A_BYTES;
          const uint32_t b_dst = sb + C::OFF_B + (uint32_t)s * C::B_BYTES;
          if constexpr (PAIR) {
            const uint32_t fb = full0_leader + 8u * (uint32_t)s;
            tma_load_2d_pair(a_dst, mA, fb, kb * C::BK, ay);
#pragma unroll
            for (int j = 0; j < C::B_BOXES; ++j)
              tma_load_2d_pair(b_dst + j * C::BK * 128, mB, fb, bx + 64 * j, kb * C::BK);
          } else {
            const uint32_t fb = bar(C::BAR_FULL + s);
            if constexpr (C::A_MCAST)   // this CTA's rows of the shared A tile, to its whole row
              tma_load_2d_multicast(a_dst + (uint32_t)(rn * C::A_OWN_ROWS * C::A_ROW), mA, fb, kb * C::BK,
                                    a_row0, row_ctas);
            else
              tma_load_2d(a_dst, mA, fb, kb * C::BK, ay);
#pragma unroll
            for (int i = 0; i < C::B_OWN_BOXES; ++i) {
              const int j = rm * C::B_OWN_BOXES + i;   // this CTA's share of the B tile
              if constexpr (C::MCAST)
                tma_load_2d_multicast(b_dst + j * C::BK * 128, mB, fb, bx + 64 * j, kb * C::BK, col_ctas);
              else
                tma_load_2d(b_dst + j * C::BK * 128, mB, fb, bx + 64 * j, kb * C::BK);
            }
          }
          if (++s == C::STAGES) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        ++tile;
        const uint64_t t_req = p.trace ? globaltimer() : 0;
        w = it.next(p, rank, sb, ctl, false);
        if (p.trace && w.valid && !w.skip) p.trace[TRACE_WORDS * (size_t)w.pos + 4] = globaltimer() - t_req;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if ((!PAIR || rank == 0) && elect_one()) {
      WorkIter<BN, CL, PAIR, SCHED, RN> it;
      Work w = it.first(p, rank);
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      constexpr uint32_t idesc = make_idesc<C::MMA_M, BN>();
      constexpr uint16_t all_ctas = (uint16_t)((1u << CL) - 1u);
      while (w.valid) {
        if (kBoundsCheck && w.skip) {
          w = it.next(p, rank, sb, ctl, false);
          continue;
        }
        if (!bar_wait<PAIR>(bar(C::BAR_ACC_EMPTY + acc), aph ^ 1, p, ctl, WAIT_ACC_EMPTY)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < w.kb; ++kb) {
          if (!bar_wait(bar(C::BAR_FULL + s), ph, p, ctl, WAIT_FULL)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = sb + C::OFF_A + (uint32_t)s * C::A_BYTES;
          const uint32_t b_addr = sb + C::OFF_B + (uint32_t)s * C::B_BYTES;
#pragma unroll
          for (int kk = 0; kk < C::BK / UMMA_K; ++kk)
            mma_bf16<C::CG>(d, desc_a<C>(a_addr + kk * UMMA_K * 2), desc_b<C>(b_addr + kk * UMMA_K * 128), idesc,
                            (kb | kk) != 0);
          // the stage is free once these MMAs have read it: in every CTA that shares it
          if constexpr (PAIR) mma_commit_pair(bar(C::BAR_EMPTY + s), 0x3);
          else if constexpr (C::MCAST) mma_commit_multicast(bar(C::BAR_EMPTY + s), all_ctas);
          else mma_commit(bar(C::BAR_EMPTY + s));
          if (++s == C::STAGES) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        if constexpr (PAIR) mma_commit_pair(bar(C::BAR_ACC_FULL + acc), 0x3);
        else mma_commit(bar(C::BAR_ACC_FULL + acc));
        if (p.trace) p.trace[TRACE_WORDS * (size_t)w.pos + 7] = globaltimer();
        acc ^= 1;
        if (acc == 0) aph ^= 1;
        w = it.next(p, rank, sb, ctl, false);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ CLC scheduler
    if (SCHED == SCHED_CLC && rank == 0 && !p.hold_scheduler && elect_one()) {
      int s = 0;
      uint32_t ph = 0;
      for (int r = 0;; ++r) {
        // throttle: fetch for tile r+1 only once the producer has started tile r
        const int t = r % THR_DEPTH;
        if (!bar_wait(bar(C::BAR_THR_FULL + t), (r / THR_DEPTH) & 1, p, ctl, WAIT_THR_FULL)) break;
        mbar_arrive(bar(C::BAR_THR_EMPTY + t));
        // producer acquire: every consumer has released this response slot
        if (!bar_wait<(CL > 1)>(bar(C::BAR_CLC_EMPTY + s), ph ^ 1, p, ctl, WAIT_CLC_EMPTY)) break;
        const uint32_t full = bar(C::BAR_CLC_FULL + s);
        const uint32_t resp = sb + C::OFF_RESP + 16u * (uint32_t)s;
        const bool inject = p.inject_fail_after >= 0 && r >= p.inject_fail_after;
        const uint64_t t_issue = p.trace ? globaltimer() : 0;
        if (!inject) {
          mbar_arrive_expect_tx(full, 16);
          if constexpr (CL == 1) {
            clc_try_cancel(resp, full);
          } else {
            // every CTA of the cluster receives the response at the same offset
#pragma unroll
            for (uint32_t rk = 1; rk < (uint32_t)CL; ++rk) mbar_arrive_expect_tx_cluster(map_to_rank(full, rk), 16);
            clc_try_cancel_all(resp, full);
          }
        } else {
          // test hook: report a failed fetch without issuing a cancel
          misc[2 + s] = 1;
          mbar_arrive(full);
#pragma unroll
          for (uint32_t rk = 1; rk < (uint32_t)CL; ++rk) {
            const uint32_t peer_flag = map_to_rank(smem_addr((const void*)(misc + 2 + s)), rk);
            asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_flag), "r"(1u) : "memory");
            mbar_arrive_cluster(map_to_rank(full, rk));
          }
        }
        // the scheduler consumes the response too: it stops at the first failure
        bool ok = false;
        if (bar_wait(full, ph, p, ctl, WAIT_CLC_FULL)) {
          uint32_t x = 0;
          if (misc[2 + s] == 0) ok = clc_decode(resp, x);
          fence_proxy_async_smem();
          if (ok && p.trace) {
            const Work got = make_work<CL, RN>(p, (int)(x / C::CLX), 0);
            if (got.valid && !got.skip) p.trace[TRACE_WORDS * (size_t)got.pos + 5] = globaltimer() - t_issue;
          }
        }
        mbar_arrive(bar(C::BAR_CLC_EMPTY + s));
        if (++s == CLC_DEPTH) { s = 0; ph ^= 1; }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp >= EPI_WARP0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp - EPI_WARP0;   // TMEM lane quadrant (warp % 4)
    WorkIter<BN, CL, PAIR, SCHED, RN> it;
    Work w = it.first(p, rank);
    int acc = 0;
    uint32_t aph = 0;
    bool first_tile = true;
    const uint32_t cbuf = sb + C::OFF_C + (uint32_t)q * (uint32_t)C::C_BUFS * C::C_BUF_BYTES;
    const uint32_t acc_empty_leader0 = PAIR ? map_to_rank(bar(C::BAR_ACC_EMPTY), 0) : bar(C::BAR_ACC_EMPTY);
    int chunk_seq = 0;
    while (w.valid) {
      // The tile after this one, taken before this one is drained (its response was fetched
      // a tile ago): none means this is the CTA's last tile.  A wait that runs out here
      // still lets the current tile be drained: its accumulator completes on its own.
      const Work nxt = it.next(p, rank, sb, ctl, true);
      if (kBoundsCheck && w.skip) {
        w = nxt;
        continue;
      }
      if (!bar_wait(bar(C::BAR_ACC_FULL + acc), aph, p, ctl, WAIT_ACC_FULL)) break;
      tc_fence_after();
      if (p.trace && q == 0 && lane == 0) p.trace[TRACE_WORDS * (size_t)w.pos + 6] = globaltimer();
      const CUtensorMap* mC = p.G ? p.gmaps + 3 * w.g + 2 : &p.tmC;
      const uint32_t tcol = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      // Last tile: the producer has issued its final load and the accumulator is complete, so
      // every MMA that read the ring has finished and the whole ring is free.  Not after a
      // wait of this CTA ran out: then "no next tile" may be this warp's own timeout, and
      // the ring is left alone.
      // (Decided by lane 0 for the whole warp: the flag may change while lanes read it.)
      const bool ring_stage =
          __shfl_sync(0xffffffffu, (int)(C::RING_STAGING && !nxt.valid && *ctl.abort == 0), 0) != 0;
      if (ring_stage) fence_proxy_async_smem();   // the ring was last written by TMA loads
#pragma unroll 1
      for (int ch = 0; ch < BN / C::EPI_CHUNK; ++ch) {
        uint32_t v[C::EPI_CHUNK];
        if constexpr (C::EPI_CHUNK == 32) tmem_ld_32x32b_x32(tcol + (uint32_t)(ch * C::EPI_CHUNK), v);
        else tmem_ld_32x32b_x16(tcol + (uint32_t)(ch * C::EPI_CHUNK), v);
        tmem_wait_ld();
        if (ch == BN / C::EPI_CHUNK - 1) {
          // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (!PAIR) mbar_arrive(bar(C::BAR_ACC_EMPTY + acc));
            else mbar_arrive_cluster(acc_empty_leader0 + 8u * (uint32_t)acc);
          }
        }
        if (w.kb == 0) {
#pragma unroll
          for (int j = 0; j < C::EPI_CHUNK; ++j) v[j] = 0u;
        }
        const uint32_t buf = ring_stage ? sb + C::OFF_A + (uint32_t)(q * C::CHUNKS + ch) * C::C_BUF_BYTES
                                        : cbuf + (uint32_t)(chunk_seq % C::C_BUFS) * C::C_BUF_BYTES;
        // the store that last used `buf` has finished reading it (a ring buffer is used once)
        if (!ring_stage && lane == 0) bulk_wait_group_read<C::C_BUFS - 1>();
        __syncwarp();
        // row `lane` of the box; TMA swizzle: 16-byte chunk j of a 128-byte row sits at
        // j ^ (row % 8), of a 64-byte row at j ^ ((row / 2) % 4)
        const uint32_t row = buf + lane * (uint32_t)C::C_ROW;
        const uint32_t xr = (C::C_ROW == 128) ? (lane & 7u) : ((lane >> 1) & 3u);
#pragma unroll
        for (int j = 0; j < C::C_ROW / 16; ++j) {
          const uint32_t dst = row + (((uint32_t)j ^ xr) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v[4 * j]), "r"(v[4 * j + 1]),
                       "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(mC, buf, w.n_blk * BN + ch * C::EPI_CHUNK, w.m_blk * BM + q * 32);
          bulk_commit_group();
        }
        ++chunk_seq;
      }
      if (q == 0 && lane == 0) {
        if (p.log_owner) {
          p.log_owner[w.pos] = worker;
          log_claim(p.log_claims + w.pos, p.log_epoch);
          if (first_tile && rank == 0) {
            if (kBoundsCheck && (worker < 0 || (long long)worker >= p.n_workers)) report_bounds(p, CHK_WORKER);
            else p.log_first[worker] = ((unsigned long long)p.log_epoch << 32) | (unsigned)w.c;
          }
        }
        if (p.trace) {
          p.trace[TRACE_WORDS * (size_t)w.pos + 1] = globaltimer();
          p.trace[TRACE_WORDS * (size_t)w.pos + 2] = smid();
          p.trace[TRACE_WORDS * (size_t)w.pos + 3] = (unsigned long long)worker;
        }
      }
      first_tile = false;
      acc ^= 1;
      if (acc == 0) aph ^= 1;
      w = nxt;
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  if constexpr (CL > 1) cluster_sync(); else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<C::CG>(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace clcg
