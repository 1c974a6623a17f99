// gp_internal.h -- declarations shared by the host API and the kernel
// translation units of the pipelined GEMM library.  Not installed; the public
// interface is include/gemm_pipelined.h.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_pipelined.h"

namespace gp {

// ---------------------------------------------------------------------------
// per-call status
// ---------------------------------------------------------------------------
// Every call gets a nonzero 32-bit id and one slot of a per-device ring of
// kStatusSlots 64-bit words (slot = id mod kStatusSlots).  A kernel that gives
// up a wait stores {id, code | site << 8} there (the first error of the call
// wins; a record of another call in the slot is overwritten).  The host reads
// the slot on the call's own stream and takes a record as this call's only if
// its id matches, so slots never need clearing and concurrent calls on other
// streams cannot report or clear each other's errors.
constexpr uint32_t kDevErrTimeout = 1;  // a bounded wait gave up
constexpr int kStatusSlots = 4096;

// wait-site codes (bits 8.. of a status record) -- which wait gave up
enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteConsumerFull = 2,
  kSiteMmaAccEmpty = 3,
  kSiteEpilogueAccFull = 4,
  kSitePingPongMma = 5,
  kSiteDrain = 6,
  kSiteConvReady = 7,     // INT8 overlap engine: producer waiting for a K step's FP16 copies
  kSiteConvRing = 8,      // INT8 overlap engine: converter / signaller hand-off
  kSiteKSplitXfer = 9,    // K split over two pairs: accumulator hand-off between the pairs
};

struct KernelCtl {
  unsigned long long* status;   // this call's status slot (see kStatusSlots)
  uint32_t call_id;             // tag of this call's records in it
  uint64_t timeout_ns;      // limit of every bounded wait
  int32_t inject_lost_load; // test hook: producer skips the final tile load
  int32_t inputs_ready;     // FP16/BF16 ring: the caller promised that nothing in flight writes A or B,
                            // so loads and MMAs may start before the previous kernel has completed
};

// Stream-K split of a persistent launch over W workers (CTAs, or CTA pairs):
// the first dp_tiles output tiles (in raster order) are computed whole,
// worker w taking tiles w, w+W, ...; the K-loops of the next sk_tiles tiles
// form sk_tiles*k_tiles units of one K step each, dealt out as W contiguous,
// equal ranges.  Every segment of a tile split that way stores its FP32
// partial accumulator in the workspace (slot (2w + j) * CTAs-per-worker +
// rank, j = 0 for a worker's first segment, 1 for its last) and counts itself
// on the tile's 64-bit counter {epoch, count}; the segment that brings the
// count to the number of segments sums every partial in K order and writes C.
// Nothing waits on another CTA, so no co-residency is required.
struct SkParams {
  int32_t dp_tiles;
  int32_t sk_tiles;
  float* workspace;         // 2 * grid partial tiles, 128 x BN FP32 each
  uint32_t* flags;          // sk_tiles * CTAs-per-worker 64-bit counters (as 32-bit word pairs)
  uint32_t epoch;           // tag of this launch's counts
  int32_t raster_gm;        // M blocks per group of the tile raster (gp_plan.raster_gm)
  int32_t b_resident;       // contiguous tile ranges per worker, B kept in the ring (gp_plan.b_resident)
};

// FP32 FFMA path, K-loop split over k_splits CTAs per tile (plan.k_splits):
// CTA b computes tile b % tiles over the K steps of split b / tiles.  With
// more than one split each CTA stores its 128 x 128 FP32 partial in slot
// tile * splits + split and counts itself on the tile's {epoch, count}
// counter; the last one adds the partials in split order and writes C.
struct FfmaSplit {
  int32_t splits;
  float* workspace;
  unsigned long long* counters;
  uint32_t epoch;
};

// ---------------------------------------------------------------------------
// shared-memory budget
// ---------------------------------------------------------------------------
constexpr int kSmemPerCtaMax = 232448;   // 227 KB opt-in dynamic shared memory per CTA on sm_100/sm_103
constexpr int kSmemAlignSlack = 1024;    // dynamic smem base is re-aligned to 1024 B (128-byte swizzle atoms)
constexpr int kBarrierRegion = 256;      // mbarriers, TMEM address slot, abort flag
constexpr int kMaxStages = 8;

// FFMA (FP32) family: CTA tile 128 x 128 x 8, 8 compute warps, 8x8 outputs per thread.
constexpr int kFfmaBM = 128, kFfmaBN = 128, kFfmaBK = 8;
constexpr int kFfmaStageBytes = (kFfmaBM * kFfmaBK + kFfmaBK * kFfmaBN) * 4;
// The TMA ring takes 32 K steps per slot up to 6 slots and 16 for 7-8 (so
// that 8 slots still fit): fewer slot hand-offs per FMA than 8 (measured at
// FP32 1024^3: 35.6 TFLOP/s with 8, 38.6 with 16, 40.1 with 32).  The
// register-staged baselines keep the 8 their thread-to-element mapping is
// built for.  A K-loop shared by several CTAs is cut every kFfmaSplitK K
// steps in every variant, so all of them add the same partial sums.
constexpr int kFfmaSplitK = 32;
constexpr int ffma_ring_bk(int stages) { return stages <= 6 ? 32 : 16; }
constexpr int ffma_ring_stage_bytes(int stages) {
  return (kFfmaBM * ffma_ring_bk(stages) + ffma_ring_bk(stages) * kFfmaBN) * 4;
}

// IMMA (INT8) family: CTA tile 128 x BN x 128, BN in {128, 64}; 8 compute warps (2 x 4).
constexpr int kImmaBM = 128, kImmaBK = 128;
__host__ __device__ constexpr int imma_stage_bytes(int bn) { return (kImmaBM + bn) * kImmaBK; }

// UMMA (FP16/BF16, tcgen05) family: CTA tile 128 x BN x 64, BN in {256, 128, 64}.
constexpr int kUmmaBM = 128, kUmmaBK = 64;
constexpr int kUmmaEpiWarps = 4;
constexpr int kUmmaEpiRows = 32;         // rows per epilogue warp (one TMEM lane quarter)
constexpr int kUmmaEpiCols = 64;         // 16-bit columns per staged chunk (128 bytes)
constexpr int kUmmaEpiBufBytes = kUmmaEpiRows * kUmmaEpiCols * 2;
constexpr int kUmmaEpiBytes = kUmmaEpiWarps * 2 * kUmmaEpiBufBytes;   // double-buffered per warp
// K split over the two pairs of a cluster (256 x 128 tiles): one CTA's 128 x 128 FP32 half of the
// other pair's accumulator, received through distributed shared memory.
constexpr int kUmmaKxBytes = 128 * 128 * 4;
// CTA-pair kernel: 256 x 256 output tile per pair, 128 rows of A and of B per CTA.
constexpr int kUmmaPairStageBytes = 2 * 128 * kUmmaBK * 2;             // per CTA per K step
__host__ __device__ constexpr int umma_stage_bytes(int bn) { return (kUmmaBM + bn) * kUmmaBK * 2; }

__host__ __device__ constexpr int ring_smem_total(int ring_bytes, int extra) {
  return kSmemAlignSlack + ring_bytes + extra + kBarrierRegion;
}

// INT8 on tcgen05 with the conversion overlapped inside the GEMM kernel: the
// two-pass engine's ring and epilogue staging, an int8 staging ring of G slots
// (one conversion unit each: 128 rows x 64 int8) and the hand-off barriers.
constexpr int kI8ConvUnitBytes = 128 * 64;
constexpr int kI8MaxStg = 8;
constexpr int kI8ConvBarrierBytes = 384;
__host__ __device__ constexpr int i8_overlap_smem_total(int stages, int stg_slots) {
  return ring_smem_total(stages * kUmmaPairStageBytes + stg_slots * kI8ConvUnitBytes + kI8ConvBarrierBytes,
                         kUmmaEpiBytes);
}
// Staging slots that fit beside an S-slot ring (at most kI8MaxStg; fewer than 2: S is too deep).
__host__ __device__ constexpr int i8_overlap_staging_slots(int stages) {
  return (kSmemPerCtaMax - i8_overlap_smem_total(stages, 0)) / kI8ConvUnitBytes < kI8MaxStg
             ? (kSmemPerCtaMax - i8_overlap_smem_total(stages, 0)) / kI8ConvUnitBytes
             : kI8MaxStg;
}

// ---------------------------------------------------------------------------
// launch interface between the API and the kernel translation units
// ---------------------------------------------------------------------------
struct LaunchArgs {
  const void* A;
  const void* B;
  void* C;
  int32_t M, N, K;
  int32_t dtype, layout, variant;
  gp_plan plan;
  cudaStream_t stream;
  KernelCtl ctl;
  SkParams sk;
  FfmaSplit ks;
  int32_t ffma_tm, ffma_tn; // FFMA ring: thread tile
  void* conv;               // INT8 on tcgen05: FP16 copies of A then B, (M + N) * K halves
  bool i8_overlap;          // INT8 on tcgen05: the GEMM kernel writes the FP16 copies itself
  bool conv_early;          // INT8 two-pass: convert while the previous GEMM runs (inputs_ready)
  uint32_t* conv_ctrs;      // ... its two counter sets: {batch counter, conv_kcap K-step counters}
  int32_t conv_kcap;
  uint32_t conv_parity;     // ... the set this launch uses (it zeroes the other)
  bool one_tile;            // gp_options.one_tile_per_cta: one output tile per CTA, grid = tiles
  int32_t sm_count;
};

// Each family launcher fills *kernel with the function launched (for
// cudaFuncGetAttributes) and returns a cudaError_t.
cudaError_t launch_ffma(LaunchArgs& a, const void** kernel);
// Compute threads of the FFMA ring for thread tile tm x tn (0: that tile is not built).
int ffma_ring_compute_threads(int tm, int tn);
cudaError_t launch_imma(LaunchArgs& a, const void** kernel);
cudaError_t launch_umma(LaunchArgs& a, const void** kernel);
// CTA pairs of the pair kernel for dtype (FP16/BF16 ring, or INT8 on tcgen05: two-pass or
// conversion overlapped in the kernel) that fit at once.
cudaError_t umma_pair_capacity(int dtype, int smem_bytes, int* pairs, bool i8_overlap = false);
// Clusters of four CTAs (two pairs splitting each 256 x 128 tile's K-loop) resident at once.
cudaError_t umma_kx_capacity(int dtype, int smem_bytes, int* clusters);
// INT8 x INT8 -> INT32 on tcgen05 (FP16 operands, accumulator restarted every 1024 K).
cudaError_t launch_umma_i8(LaunchArgs& a, const void** kernel);
cudaError_t launch_zero_fill(void* C, int64_t bytes, cudaStream_t stream);

// Tensor-map encoding (driver entry point obtained once through the runtime).
// inner/outer: extents in elements; row_bytes: stride of the outer dimension.
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType type, uint64_t inner,
                         uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle swizzle);

// Opt a kernel into more than 48 KB of dynamic shared memory (cached per device).
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

}  // namespace gp
