// api.cu -- the C ABI (include/gemm_pipelined.h): argument checks, tile and
// stage selection against the shared-memory budget, tensor-map encoding,
// dispatch to the kernel families, and the per-thread last-call record.
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include <cudaTypedefs.h>

#include "gp_internal.h"

namespace gp {

// Per-call status slots, a ring per device (every device that loads the
// library holds its own copy: 32 KiB).  Call i on a device records a failed
// wait in slot i mod kStatusSlots, tagged with its id (see kStatusSlots).
__device__ unsigned long long g_status_ring[kStatusSlots];

namespace {

constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s
constexpr int kMaxDevices = 64;

// ---------------------------------------------------------------------------
// per-device caches
// ---------------------------------------------------------------------------
std::mutex g_mu;
unsigned long long* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
uint32_t g_call_id[kMaxDevices] = {};

// SM count of `dev` and, for a new call, its id and status slot.
cudaError_t device_info(int dev, int* sms, uint32_t* call_id, unsigned long long** slot) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_status_ring);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned long long*>(p);
    g_sm_count[dev] = n;
  }
  if (++g_call_id[dev] == 0) g_call_id[dev] = 1;   // 0 would match an untouched slot
  *sms = g_sm_count[dev];
  *call_id = g_call_id[dev];
  *slot = g_status_ptr[dev] + (g_call_id[dev] % kStatusSlots);
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// tensor maps
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct TmapKey {
  int dev;
  const void* base;
  int type;
  uint64_t inner, outer, row_bytes;
  uint32_t box_inner, box_outer;
  int swizzle;
  bool operator==(const TmapKey& o) const {
    return dev == o.dev && base == o.base && type == o.type && inner == o.inner && outer == o.outer &&
           row_bytes == o.row_bytes && box_inner == o.box_inner && box_outer == o.box_outer && swizzle == o.swizzle;
  }
};

struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  uint64_t stamp;
  bool used;
};

constexpr int kTmapCache = 64;
TmapEntry g_tmaps[kTmapCache];
uint64_t g_tmap_clock = 0;

// ---------------------------------------------------------------------------
// stream-K workspace: per device and stream, grown on demand, never shrunk.
// Calls on one stream are ordered, so one workspace per stream is race-free.
// The table holds kMaxWorkspaces streams; a new stream beyond that takes over
// the least recently used entry after a device-wide synchronisation (the
// entry's stream may have been destroyed, so it is not used).  gemm_release
// frees a device's workspaces.
// ---------------------------------------------------------------------------
struct Workspace {
  int dev = -1;
  cudaStream_t stream = nullptr;
  uint64_t last_use = 0;
  float* partials = nullptr;
  size_t bytes = 0;
  uint32_t* flags = nullptr;
  size_t nflags = 0;
  uint32_t epoch = 0;
  void* conv = nullptr;       // INT8 on tcgen05: FP16 copies of the operands
  size_t conv_bytes = 0;
  size_t conv_off = 0;        // region [conv_off, conv_off + conv_len) the last INT8 call on this stream used
  size_t conv_len = 0;
  uint32_t* ov_ctrs = nullptr;   // INT8 conversion / GEMM hand-off counters: two sets of ov_kcap + 1 words
  int32_t ov_kcap = 0;
  uint32_t ov_launches = 0;
};
constexpr int kMaxWorkspaces = 64;
Workspace g_ws[kMaxWorkspaces];
uint64_t g_ws_clock = 0;

// Free an entry's buffers (nothing may still use them) and mark it empty.
void free_workspace(Workspace& w) {
  if (w.partials) cudaFree(w.partials);
  if (w.flags) cudaFree(w.flags);
  if (w.conv) cudaFree(w.conv);
  if (w.ov_ctrs) cudaFree(w.ov_ctrs);
  w = Workspace();
}

// The entry of (dev, stream), created if needed.  Caller holds g_mu; dev is current.
cudaError_t find_workspace(int dev, cudaStream_t stream, Workspace** out) {
  Workspace* w = nullptr;
  for (auto& x : g_ws)
    if (x.dev == dev && x.stream == stream) { w = &x; break; }
  if (!w) {
    for (auto& x : g_ws)
      if (x.dev < 0) { w = &x; break; }
  }
  if (!w) {
    // every entry taken: reclaim the least recently used one
    Workspace* lru = &g_ws[0];
    for (auto& x : g_ws)
      if (x.last_use < lru->last_use) lru = &x;
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    const int owner = lru->dev;
    if (owner != cur && (e = cudaSetDevice(owner)) != cudaSuccess) return e;
    e = cudaDeviceSynchronize();   // whatever its stream still had in flight is done
    if (e == cudaSuccess) free_workspace(*lru);
    if (owner != cur) cudaSetDevice(cur);
    if (e != cudaSuccess) return e;
    w = lru;
  }
  if (w->dev < 0) {
    w->dev = dev;
    w->stream = stream;
  }
  w->last_use = ++g_ws_clock;
  *out = w;
  return cudaSuccess;
}

cudaError_t get_workspace(int dev, cudaStream_t stream, size_t bytes, size_t nflags, float** partials,
                          uint32_t** flags, uint32_t* epoch) {
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace* w = nullptr;
  cudaError_t e = find_workspace(dev, stream, &w);
  if (e != cudaSuccess) return e;
  if (w->bytes < bytes) {
    if (w->partials) {
      if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
      cudaFree(w->partials);
      w->partials = nullptr;
      w->bytes = 0;
    }
    if ((e = cudaMalloc(&w->partials, bytes)) != cudaSuccess) return e;
    w->bytes = bytes;
  }
  if (w->nflags < nflags) {
    if (w->flags) {
      if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
      cudaFree(w->flags);
      w->flags = nullptr;
      w->nflags = 0;
    }
    if ((e = cudaMalloc(&w->flags, nflags * sizeof(uint32_t))) != cudaSuccess) return e;
    if ((e = cudaMemset(w->flags, 0, nflags * sizeof(uint32_t))) != cudaSuccess) return e;
    w->nflags = nflags;
    w->epoch = 0;
  }
  if (++w->epoch == 0) w->epoch = 1;   // split-tile counters are tagged with the launch's epoch
  *partials = w->partials;
  *flags = w->flags;
  *epoch = w->epoch;
  return cudaSuccess;
}

// FP16 operand buffer of the INT8 tcgen05 path, per device and stream.  With
// alternate = true the call's copies must not overlap the region the previous
// call on this stream used (its conversion may run while that call's GEMM
// still reads them): they go below that region if they fit there, else above
// it, else the buffer is regrown (after the stream has drained).  Otherwise
// (conversion ordered after all earlier work) they start at offset 0.
cudaError_t get_conv_workspace(int dev, cudaStream_t stream, size_t bytes, void** conv, bool alternate = false) {
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace* w = nullptr;
  cudaError_t e0 = find_workspace(dev, stream, &w);
  if (e0 != cudaSuccess) return e0;
  constexpr size_t kAlign = 256;
  const size_t above = (w->conv_off + w->conv_len + kAlign - 1) / kAlign * kAlign;
  size_t off = 0;
  bool grow = w->conv_bytes < bytes;
  if (alternate && !grow) {
    if (w->conv_len == 0 || bytes <= w->conv_off)
      off = 0;
    else if (above + bytes <= w->conv_bytes)
      off = above;
    else
      grow = true;
  }
  if (grow) {
    cudaError_t e;
    if (w->conv) {
      if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;   // nothing reads the old buffer now
      cudaFree(w->conv);
      w->conv = nullptr;
      w->conv_bytes = 0;
    }
    const size_t cap = alternate ? 2 * (bytes + kAlign) : bytes;
    if ((e = cudaMalloc(&w->conv, cap)) != cudaSuccess) return e;
    w->conv_bytes = cap;
    off = 0;
  }
  w->conv_off = off;
  w->conv_len = bytes;
  *conv = static_cast<unsigned char*>(w->conv) + off;
  return cudaSuccess;
}

// Counters of the INT8 overlap engine, per device and stream: two sets of
// {batch counter, kcap K-step counters}, used by alternate launches (each
// launch zeroes the other set for its successor).  Zeroed when (re)allocated.
cudaError_t get_overlap_ctrs(int dev, cudaStream_t stream, int64_t k_tiles, uint32_t** ctrs, int32_t* kcap,
                             uint32_t* parity) {
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace* w = nullptr;
  cudaError_t e = find_workspace(dev, stream, &w);
  if (e != cudaSuccess) return e;
  if (w->ov_kcap < k_tiles) {
    if (w->ov_ctrs) {
      if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
      cudaFree(w->ov_ctrs);
      w->ov_ctrs = nullptr;
      w->ov_kcap = 0;
    }
    const int64_t cap = std::max<int64_t>(k_tiles, 64);
    const size_t bytes = 2 * static_cast<size_t>(cap + 1) * sizeof(uint32_t);
    if ((e = cudaMalloc(&w->ov_ctrs, bytes)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(w->ov_ctrs, 0, bytes, stream)) != cudaSuccess) return e;
    w->ov_kcap = static_cast<int32_t>(cap);
    w->ov_launches = 0;
  }
  *ctrs = w->ov_ctrs;
  *kcap = w->ov_kcap;
  *parity = (w->ov_launches++) & 1u;
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// per-thread last-call record
// ---------------------------------------------------------------------------
struct LastCall {
  gp_stats stats;
  int device = -1;
  cudaStream_t stream = nullptr;
  unsigned long long* status_slot = nullptr;   // the call's status slot and id (see kStatusSlots)
  uint32_t call_id = 0;
  const void* kernel = nullptr;
  bool timed = false;
  cudaEvent_t ev[2] = {nullptr, nullptr};
  int ev_device = -1;
  bool valid = false;
};
thread_local LastCall t_last;

int family_of(int dtype) {
  switch (dtype) {
    case GP_F32: return 0;                                   // FFMA
    case GP_I8_I32: return 1;                                // IMMA
    default: return 2;                                       // UMMA
  }
}

int in_elem_bytes(int dtype) {
  switch (dtype) {
    case GP_I8_I32: return 1;
    case GP_F32: return 4;
    default: return 2;
  }
}

int out_elem_bytes(int dtype) { return dtype == GP_I8_I32 || dtype == GP_F32 ? 4 : 2; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// FFMA: 3; IMMA: 4 (more buys nothing once the IMMA pipe is busy); tcgen05: 6
// (the deepest ring the CTA-pair tile fits in 227 KB).
// Kernel name of the FFMA ring for a thread tile (a static string).
const char* ffma_ring_name(int tm, int tn) {
  switch (tm * 100 + tn) {
    case 408: return "ffma_ring_4x8";
    case 804: return "ffma_ring_8x4";
    case 816: return "ffma_ring_8x16";
    case 1608: return "ffma_ring_16x8";
    case 1616: return "ffma_ring_16x16";
    default: return "ffma_ring";
  }
}

// INT8 engine with the int8 -> FP16 conversion in the producer warps (gp_options.i8_engine).
constexpr int kI8EngineOverlap = 3;
const char* const kI8OverlapKernelName = "umma_i8_overlap_pair_ring";
constexpr int kI8OverlapDefaultStages = 5;   // the deepest ring that leaves room for int8 staging
static_assert(i8_overlap_staging_slots(kI8OverlapDefaultStages) >= 2 &&
                  i8_overlap_staging_slots(kI8OverlapDefaultStages + 1) < 2,
              "overlap engine depth limit");

// INT8 on tcgen05: bytes of the FP16 copies of A and B.
int64_t i8_conv_bytes(int64_t M, int64_t N, int64_t K) { return (M + N) * K * 2; }

// M blocks per group of the tile raster of the persistent tcgen05 rings:
// one group over all of them when there are at most kWholeRasterBlocks and
// their A panels take at most kWholeRasterBytes (every wave then sweeps the
// whole of A, which stays in L2, while each B panel is read by one wave's
// worth of tiles at once: at FP16 4096^3, 124 against 144 MB of DRAM traffic
// per launch and 2 % less time than groups of 8), else groups of 8 (measured
// as fast or faster on 8192-row problems: BF16 8192^2 x 16384, 1166 against
// 1202 us with groups of 4).
constexpr int kDefaultRasterGM = 8;
constexpr int64_t kWholeRasterBlocks = 16;
constexpr int64_t kWholeRasterBytes = int64_t(48) << 20;
int auto_raster_gm(int64_t M, int64_t K, int bm, int in_bytes) {
  const int64_t m_blocks = (M + bm - 1) / bm;
  if (m_blocks <= kWholeRasterBlocks && M * K * in_bytes <= kWholeRasterBytes) return static_cast<int>(m_blocks);
  return kDefaultRasterGM;
}

// FP16/BF16 GEMMs with K up to this many elements run one CTA per tile, not CTA pairs.
constexpr int64_t kShortK = 256;

int default_stages(int family) { return family == 0 ? 3 : (family == 1 ? 4 : 6); }

// Persistent FP16/BF16 ring: when the output tiles do not fill whole waves of
// `workers` (CTAs, or CTA pairs), keep the full waves as whole tiles and
// spread the K steps of the rest evenly over every worker (stream-K); with a
// ring of at most kShallowSplitStages slots, the last full wave is split too.
// A split costs a partial-tile write and read plus a flag wait, a few
// microseconds; it pays only when whole-tile scheduling would leave the
// average worker idle for at least kMinIdleSteps K steps at the tail.
// Measured interleaved, with a pause between samples (FP16/BF16, CTA pairs):
// splitting only the tiles left after the full waves took the default 6-slot
// ring at 4096^2 x 8192 from 161.9 to 157.3 us and at 8192^2 x 16384 from 1181
// to 1150 us, and 4096^3 from 80.6 to 80.5 us; it also cut the DRAM reads at
// 4096^3 from 91.5 to 88.3 MB.  At 3 and 4 slots it was 2-3 % slower (96.0
// against 99.0 us, 83.8 against 85.7 us at 4096^3).
constexpr int kShallowSplitStages = 4;
void apply_stream_k(gp_plan* p, int64_t workers, int ctas_per_worker, bool allowed) {
  constexpr int64_t kMinIdleSteps = 16;
  constexpr int64_t kMinStepsPerWorker = 4;
  const int64_t T = p->tiles, G = workers;
  p->dp_tiles = static_cast<int32_t>(T);
  p->sk_tiles = 0;
  p->workspace_bytes = 0;
  p->grid = static_cast<int32_t>(ctas_per_worker * (T < G ? T : G));
  if (!allowed || G <= 0 || p->k_tiles <= 0 || T % G == 0) return;
  const int64_t idle_tiles = ((T + G - 1) / G) * G - T;        // empty slots of the last wave
  if (idle_tiles * p->k_tiles < kMinIdleSteps * G) return;
  const int64_t full_waves = T / G - (p->stages <= kShallowSplitStages ? 1 : 0);
  const int64_t dp = T > G ? full_waves * G : 0;
  const int64_t skt = T - dp;
  if (skt * p->k_tiles < kMinStepsPerWorker * G) return;
  p->dp_tiles = static_cast<int32_t>(dp);
  p->sk_tiles = static_cast<int32_t>(skt);
  p->grid = static_cast<int32_t>(ctas_per_worker * G);
  p->workspace_bytes = static_cast<int64_t>(p->grid) * 2 * 128 * p->bn * 4;   // two 128-row FP32 slots per CTA
}

// INT8 on tcgen05 (two-pass engine), whole tiles over W workers: when the last
// wave would hold r <= W/2 tiles, run those r tiles as 2r half tiles (BN/2
// wide) on 2r workers instead -- the same MMAs split along N, so no partial
// sums, and the last wave takes about half as long.
void apply_i8_halves(gp_plan* p, int64_t workers) {
  p->half_tiles = 0;
  if (workers <= 0 || p->sk_tiles > 0 || p->tiles <= workers) return;
  const int64_t r = p->tiles % workers;
  if (r == 0 || 2 * r > workers) return;
  p->half_tiles = static_cast<int32_t>(r);
  p->dp_tiles = static_cast<int32_t>(p->tiles - r);
}

// Tile/stage choice.  sm_count <= 0: no device queried (grid left 0 for persistent kernels).
int plan_impl(int64_t M, int64_t N, int64_t K, int dtype, int layout, int stages, int variant, int bn_req,
              int sm_count, gp_plan* p, bool no_stream_k = false, bool no_pair = false, int i8_engine = 0,
              int ffma_tm = 0, int ffma_tn = 0, int pair_k_split = 0, bool one_tile = false, int raster_gm = 0) {
  if (dtype < GP_I8_I32 || dtype > GP_F32) return GP_ERR_ARG;
  if (layout != GP_A_ROW_B_COL && layout != GP_A_ROW_B_ROW) return GP_ERR_ARG;
  if (variant < GP_PINGPONG || variant > GP_NOPIPE) return GP_ERR_ARG;
  if (M < 0 || N < 0 || K < 0) return GP_ERR_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GP_ERR_SIZE;
  if (bn_req < 0 || raster_gm < 0) return GP_ERR_ARG;
  const int fam = family_of(dtype);
  if (fam == 0 && layout != GP_A_ROW_B_ROW) return GP_ERR_UNSUPPORTED;
  if (fam != 0 && layout != GP_A_ROW_B_COL) return GP_ERR_UNSUPPORTED;

  int S;
  if (variant == GP_NOPIPE) {
    if (stages != 0 && stages != 1) return GP_ERR_ARG;
    S = 1;
  } else if (variant == GP_PINGPONG) {
    if (stages != 0 && stages != 2) return GP_ERR_ARG;
    S = 2;
  } else {
    if (stages < 0 || stages > kMaxStages) return GP_ERR_ARG;
    S = stages == 0 ? default_stages(fam) : stages;
    // FP16/BF16 with only a few K steps (K <= kShortK): one CTA per 128 x 256
    // tile beats the CTA pair (measured at 8192 x 8192 x 256, where C's write
    // dominates); its widest tile fits 4 stages.
    if (stages == 0 && family_of(dtype) == 2 && K <= kShortK && N > 128) S = 4;
    // (The 256 x 256 pair tile keeps the default 6 stages at every K: measured
    // back to back with a pause between interleaved samples, 6 against 5
    // stages took FP16 4096^3 79.5 against 80.0 us, 4096^2 x 8192 160.9
    // against 162.8 us, BF16 8192^2 x 4096 285.1 against 287.0 us, 8192^2 x
    // 8192 572.0 against 575.6 us, and 8192^2 x 16384 1155 against 1152 us.)
    // 64 < N <= 128 (the 256 x 128 pair tile, 24 KB per stage): the operand
    // stream bounds these GEMMs, so keep as many bytes in flight as fit.
    if (stages == 0 && family_of(dtype) == 2 && N > 64 && N <= 128 && M > 128 && K > kShortK) S = kMaxStages;
  }

  std::memset(p, 0, sizeof(*p));
  p->k_splits = 1;
  p->raster_gm = raster_gm > 0 ? raster_gm : kDefaultRasterGM;   // (the tcgen05 tiles refine the default below)
  p->dtype = dtype;
  p->layout = layout;
  p->variant = variant;
  p->stages = S;
  const bool ring = variant == GP_PIPELINED;

  if (i8_engine < 0 || i8_engine > 3) return GP_ERR_ARG;
  if (pair_k_split < -1 || pair_k_split > 1) return GP_ERR_ARG;
  if (pair_k_split == 1 && (fam != 2 || !ring)) return GP_ERR_UNSUPPORTED;   // FP16/BF16 ring only
  const int i8_tc_stages = stages == 0 ? 6 : S;
  if (fam == 1 && ring && i8_engine != 1 && !no_pair && !one_tile && (bn_req == 0 || bn_req == 256) &&
      ring_smem_total(i8_tc_stages * kUmmaPairStageBytes, kUmmaEpiBytes) <= kSmemPerCtaMax) {
    // INT8 on tcgen05: FP16 operands, CTA pair per 256 x 256 tile.
    // Deeper rings than this tile allows (7, 8 stages) run on the IMMA ring.
    // The overlap engine numbers its conversion units (K step x 128-row panel) in 31 bits.
    const int64_t conv_units = ceil_div(K, kUmmaBK) * (ceil_div(M, 128) + ceil_div(N, 128));
    // It also stages int8 tiles in shared memory: deeper rings than kI8OverlapDefaultStages
    // leave no room, and the two-pass engine runs them.
    const bool overlap = i8_engine == kI8EngineOverlap && conv_units < (int64_t(1) << 30) &&
                         (stages == 0 || i8_overlap_staging_slots(S) >= 2);
    S = overlap && stages == 0 ? kI8OverlapDefaultStages : i8_tc_stages;
    p->stages = S;
    p->bm = 256;
    p->bn = 256;
    p->bk = kUmmaBK;
    p->threads = overlap ? 512 : 64 + 32 * 8;
    p->stage_bytes = kUmmaPairStageBytes;
    p->ring_bytes = S * p->stage_bytes;
    p->smem_bytes = overlap ? i8_overlap_smem_total(S, i8_overlap_staging_slots(S))
                            : ring_smem_total(p->ring_bytes, kUmmaEpiBytes);
    if (p->smem_bytes < kSmemPerCtaMax / 2 + 1024) p->smem_bytes = kSmemPerCtaMax / 2 + 1024;
    p->tmem_cols = 512;
    p->persistent = 1;
    p->cta_pair = 1;
    p->kernel = overlap ? kI8OverlapKernelName : "umma_i8_pair_ring";
    p->tiles = ceil_div(M, p->bm) * ceil_div(N, p->bn);
    p->k_tiles = ceil_div(K, p->bk);
    if (p->tiles > INT32_MAX) return GP_ERR_SIZE;
    if (raster_gm <= 0) p->raster_gm = auto_raster_gm(M, K, p->bm, 2);   // the FP16 copies are what is read
    p->grid = sm_count > 1 ? static_cast<int32_t>(2 * (p->tiles < sm_count / 2 ? p->tiles : sm_count / 2)) : 0;
    p->dp_tiles = static_cast<int32_t>(p->tiles);
    p->sk_tiles = 0;
    p->workspace_bytes = 0;
    // Stream-K over the CTA pairs (int32 partials: exact in any order), only
    // when the tiles do not fill one wave: with a partial last wave the
    // heavier int32 split epilogue measured slower than whole tiles.
    // (The overlap engine writes the same FP16 copies from inside the GEMM kernel; whole tiles only.)
    if (!overlap && sm_count > 1 && p->tiles < sm_count / 2) apply_stream_k(p, sm_count / 2, 2, !no_stream_k);
    if (!overlap && sm_count > 1) apply_i8_halves(p, sm_count / 2);
    p->workspace_bytes += i8_conv_bytes(M, N, K);   // FP16 copies of A and B, after the partial tiles
    // per CTA: 128 x 256 outputs from 128 rows of A and 128 rows of B (FP16)
    p->compute_load_ratio = 2.0 * 128 * 256 * p->bk / ((128.0 + 128.0) * p->bk * 2.0);
    return GP_OK;
  }

  int cands[3] = {0, 0, 0};
  int ncand = 0;
  int extra = 0;
  if (fam == 0) {
    p->bm = kFfmaBM;
    p->bk = ring ? ffma_ring_bk(S) : kFfmaBK;
    cands[ncand++] = kFfmaBN;
    // thread tile of the ring (the register-staged variants build the pages' 8 x 8 only)
    const int tm = ffma_tm ? ffma_tm : 8, tn = ffma_tn ? ffma_tn : 8;
    const int compute_threads = ffma_ring_compute_threads(tm, tn);
    if (ring ? compute_threads == 0 : (tm != 8 || tn != 8)) return GP_ERR_UNSUPPORTED;
    p->threads = ring ? compute_threads + 32 : 256;
    p->kernel = ring ? ffma_ring_name(tm, tn) : (variant == GP_PINGPONG ? "ffma_pingpong" : "ffma_nopipe");
  } else if (fam == 1) {
    p->bm = kImmaBM;
    p->bk = kImmaBK;
    cands[ncand++] = 128;
    cands[ncand++] = 64;
    p->threads = ring ? 288 : 256;
    p->kernel = ring ? "imma_ring" : (variant == GP_PINGPONG ? "imma_pingpong" : "imma_nopipe");
  } else {
    p->bm = kUmmaBM;
    p->bk = kUmmaBK;
    cands[ncand++] = 256;
    cands[ncand++] = 128;
    cands[ncand++] = 64;
    extra = kUmmaEpiBytes;
    p->threads = ring ? 192 : 256;
    p->kernel = ring ? "umma_ring" : (variant == GP_PINGPONG ? "umma_pingpong" : "umma_nopipe");
  }
  auto stage_bytes = [&](int bn) {
    if (fam == 0) return ring ? ffma_ring_stage_bytes(S) : kFfmaStageBytes;
    if (fam == 1) return imma_stage_bytes(bn);
    return umma_stage_bytes(bn);
  };
  auto fits = [&](int bn) { return ring_smem_total(S * stage_bytes(bn), extra) <= kSmemPerCtaMax; };

  // CTA pairs (FP16/BF16 ring): a 256 x 256 tile per pair while S stages of 32 KB fit, else a
  // 256 x 128 tile (24 KB per CTA per K step, up to 8 stages) -- also the tile for 64 < N <= 128.
  auto pair_fits = [&](int pbn) {
    return ring_smem_total(S * (kUmmaBM + pbn / 2) * kUmmaBK * 2, kUmmaEpiBytes) <= kSmemPerCtaMax;
  };
  const bool pair_base = fam == 2 && ring && !no_pair && !one_tile && K > kShortK;
  const bool pair256 = pair_base && (bn_req == 0 || bn_req == 256) && N > 128 && pair_fits(256);
  const bool pair128 = pair_base && !pair256 && bn_req == 0 && N > 64 && M > 128 && pair_fits(128);
  // pair_k_split: a cluster of two pairs splits each 256 x 128 tile's K-loop
  // in two halves and adds them through distributed shared memory (for few
  // tiles and long K-loops, instead of stream-K partial tiles in L2); its
  // 64 KB receive buffer leaves room for at most 5 stages.
  const int kx_S = stages == 0 ? 5 : S;
  const bool kx_able = pair128 && ceil_div(K, kUmmaBK) >= 2 && (sm_count == 0 || sm_count >= 8) &&
                       ring_smem_total(kx_S * (kUmmaBM + 64) * kUmmaBK * 2, kUmmaEpiBytes + kUmmaKxBytes) <=
                           kSmemPerCtaMax;
  if (pair_k_split == 1 && !kx_able) return GP_ERR_UNSUPPORTED;
  // By default where the tiles about fill the clusters of four (more than
  // SMs/8, at most SMs/4) and the K-loops are long: measured at BF16 8192 x
  // 128 x 8192 (32 tiles), 32.3 us against 38.1 us with stream-K over 76
  // pairs.  Fewer tiles keep stream-K, which spreads them over more SMs.
  const int64_t kx_tiles = ceil_div(M, 256) * ceil_div(N, 128);
  const bool kx_default = sm_count > 0 && kx_tiles > sm_count / 8 && kx_tiles <= sm_count / 4 &&
                          ceil_div(K, kUmmaBK) >= 32;
  const bool kx = kx_able && (pair_k_split == 1 || (pair_k_split == 0 && kx_default));
  if (kx) {
    S = kx_S;
    p->stages = S;
  }
  const bool pair_ok = pair256 || pair128;
  const int pair_bn = pair256 ? 256 : 128;
  int bn = 0;
  if (pair_ok) {
    bn = pair_bn;   // the pair kernel below replaces the single-CTA fields
  } else if (bn_req) {
    bool known = false;
    for (int i = 0; i < ncand; ++i) known |= (cands[i] == bn_req);
    if (!known) return GP_ERR_UNSUPPORTED;
    if (!fits(bn_req)) return GP_ERR_SMEM;
    bn = bn_req;
  } else {
    for (int i = 0; i < ncand; ++i) {
      const int c = cands[i];
      const bool smaller_covers = (i + 1 < ncand) && (c / 2 >= N);
      if (fits(c) && !smaller_covers) { bn = c; break; }
    }
    if (!bn) {
      for (int i = 0; i < ncand; ++i)
        if (fits(cands[i])) { bn = cands[i]; break; }
    }
    if (!bn) return GP_ERR_SMEM;
  }
  p->bn = bn;
  p->stage_bytes = pair_ok ? (kUmmaBM + pair_bn / 2) * kUmmaBK * 2 : stage_bytes(bn);
  p->ring_bytes = S * p->stage_bytes;
  p->smem_bytes = ring_smem_total(p->ring_bytes, extra);
  if (fam == 2) {
    p->tmem_cols = ring ? 2 * bn : bn;
    if (ring && p->smem_bytes < kSmemPerCtaMax / 2 + 1024) {
      // a persistent CTA holds 2*BN TMEM columns for its whole life: keep one CTA per SM
      p->smem_bytes = kSmemPerCtaMax / 2 + 1024;
    }
  }
  p->persistent = (ring && fam != 0 && !one_tile) ? 1 : 0;
  // FP16/BF16 ring on CTA pairs: 256 x BN tile per pair; per CTA per K step 128 rows of A and
  // BN/2 rows of B (32 KB for BN 256, 24 KB for BN 128)
  if (pair_ok) {
    p->cta_pair = 1;
    p->bm = 256;
    p->bn = pair_bn;
    p->stage_bytes = (kUmmaBM + pair_bn / 2) * kUmmaBK * 2;
    p->ring_bytes = S * p->stage_bytes;
    p->smem_bytes = ring_smem_total(p->ring_bytes, kUmmaEpiBytes);
    if (p->smem_bytes < kSmemPerCtaMax / 2 + 1024) p->smem_bytes = kSmemPerCtaMax / 2 + 1024;
    p->tmem_cols = 2 * pair_bn;
    p->kernel = "umma_pair_ring";
    if (kx) {
      p->cta_pair = 3;
      p->kernel = "umma_pair_ksplit_ring";
      p->smem_bytes = ring_smem_total(p->ring_bytes, kUmmaEpiBytes + kUmmaKxBytes);
    }
  }
  p->tiles = ceil_div(M, p->bm) * ceil_div(N, p->bn);
  p->k_tiles = ceil_div(K, p->bk);
  if (p->tiles > INT32_MAX) return GP_ERR_SIZE;
  if (fam == 2 && ring && raster_gm <= 0) p->raster_gm = auto_raster_gm(M, K, p->bm, in_elem_bytes(dtype));
  if (p->cta_pair == 3)
    p->grid = sm_count > 3 ? static_cast<int32_t>(4 * (p->tiles < sm_count / 4 ? p->tiles : sm_count / 4)) : 0;
  else if (p->cta_pair)
    p->grid = sm_count > 1 ? static_cast<int32_t>(2 * (p->tiles < sm_count / 2 ? p->tiles : sm_count / 2)) : 0;
  else if (p->persistent)
    p->grid = sm_count > 0 ? static_cast<int32_t>(p->tiles < sm_count ? p->tiles : sm_count) : 0;
  else
    p->grid = static_cast<int32_t>(p->tiles);
  p->dp_tiles = static_cast<int32_t>(p->tiles);
  p->sk_tiles = 0;
  p->workspace_bytes = 0;
  if (fam == 0 && sm_count > 0 && p->tiles % sm_count != 0 && !no_stream_k && !one_tile) {
    // FFMA: the tiles do not fill whole waves of one CTA per SM.  Where the
    // whole tiles would leave SMs idle (at most 3/4 of the SMs busy in one
    // wave, or a part-empty last wave), the tiles' K-loops, laid end to end
    // in units of kFfmaSplitK K steps, are dealt out as equal contiguous
    // ranges to one CTA per SM (fewer CTAs when a range would be shorter than
    // kFfmaMinSplitSteps units).  A range meets a tile at most at its two
    // ends; the CTA that completes a shared tile adds its partial sums in K
    // order, so the result does not depend on timing, and every variant takes
    // the same ranges.  Measured (32 K steps per slot, interleaved, against
    // whole tiles or two CTAs per tile): 1024^3 51.04 -> 50.66 us; 512 x 512 x
    // 4096 96.1 -> 53.4 us; 1280^2 x 2048 (100 tiles) 173.8 -> 128.4 us;
    // 2048^3 344.9 -> 304.0 us; 4096^3 2392.5 -> 2332.4 us.  At 144 tiles on
    // 152 SMs whole tiles were 1.4 % faster.  (With 8 K steps per slot, one
    // range per SM had measured slower than whole CTAs per tile.)
    constexpr int64_t kFfmaMinSplitSteps = 256 / kFfmaSplitK;   // units of kFfmaSplitK K steps: 256 K steps
    const int64_t units = ceil_div(K, kFfmaSplitK) * p->tiles;
    int64_t grid = units / kFfmaMinSplitSteps;
    if (grid > sm_count) grid = sm_count;
    const bool few = 4 * p->tiles <= 3 * sm_count && grid > p->tiles;
    const bool waves = p->tiles > sm_count && grid == sm_count;
    if (few || waves) {
      p->grid = static_cast<int32_t>(grid);
      // CTAs sharing a tile: about grid / tiles of them when ranges are shorter than a
      // K-loop, at most two when they are longer
      p->k_splits = static_cast<int32_t>(few ? ceil_div(grid, p->tiles) : 2);
      p->workspace_bytes = 2 * grid * p->bm * p->bn * 4;   // two FP32 partial slots per CTA
    }
  }
  if (fam == 2 && ring && sm_count > 0 && !one_tile) {
    if (p->cta_pair == 3)
      ;   // whole tiles, each K-loop split over the cluster's two pairs
    else if (p->cta_pair)
      apply_stream_k(p, sm_count / 2, 2, !no_stream_k);
    else
      apply_stream_k(p, sm_count, 1, !no_stream_k);
  }
  // One-CTA ring whose whole K-loop fits the ring, on whole tiles, with more
  // tiles than CTAs: give each CTA a contiguous run of tiles in M-block-
  // fastest order and keep the B tile in the ring while the N block repeats,
  // so a tile loads only its A rows (BM x K) instead of A and B.  The ring
  // then has one slot per K step.  Measured at BF16 8192 x 8192 (back to
  // back, interleaved; bit-identical results): K = 256 34.7 -> 31.6 us, K =
  // 192 30.8 -> 28.8 us, K = 128 28.9 -> 28.4 us; FP16 4096^2 x 256 12.43 ->
  // 12.24 us.  A single K step (one slot, no load overlapping the previous
  // tile's MMAs) measured 0.4 % slower, so it keeps the streamed ring.
  if (fam == 2 && ring && !p->cta_pair && p->persistent && raster_gm <= 0 && p->sk_tiles == 0 && p->grid > 0 &&
      p->tiles > p->grid && p->k_tiles >= 2 && (p->k_tiles == S || (stages == 0 && p->k_tiles < S))) {
    p->b_resident = 1;
    p->stages = static_cast<int32_t>(p->k_tiles);
    p->ring_bytes = p->stages * p->stage_bytes;
    p->smem_bytes = ring_smem_total(p->ring_bytes, extra);
    if (p->smem_bytes < kSmemPerCtaMax / 2 + 1024) p->smem_bytes = kSmemPerCtaMax / 2 + 1024;
    p->raster_gm = static_cast<int32_t>(ceil_div(M, p->bm));
  }
  const double e = in_elem_bytes(dtype);
  p->compute_load_ratio = 2.0 * p->bm * p->bn * p->bk / ((static_cast<double>(p->bm) * p->bk + p->bk * p->bn) * e);
  if (p->cta_pair)   // per CTA: 128 x 256 outputs from 128 rows of A and 128 rows of B
    p->compute_load_ratio = 2.0 * (p->bm / 2) * p->bn * p->bk / ((p->bm / 2 + p->bn / 2) * p->bk * e);
  return GP_OK;
}

int alignment_ok(const void* A, const void* B, const void* C, int64_t N, int64_t K, int dtype) {
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                         reinterpret_cast<uintptr_t>(C)) & 15u;
  if (mis) return 0;
  switch (dtype) {
    case GP_I8_I32: return (K % 16 == 0) && (N % 4 == 0);
    case GP_F32: return (K % 4 == 0) && (N % 4 == 0);
    default: return (K % 8 == 0) && (N % 8 == 0);
  }
}

// Step of the call whose CUDA call failed (a GP_SITE_* code); helpers that run
// inside the kernel-family launchers set it when they fail.
thread_local int t_fail_site = 0;

void record(int status, int cuda_err, int site = 0) {
  t_last.stats.status = status;
  t_last.stats.cuda_error = cuda_err;
  t_last.stats.cuda_error_site = cuda_err ? site : 0;
  t_last.valid = true;
}

}  // namespace

// ---------------------------------------------------------------------------
// helpers used by the kernel translation units
// ---------------------------------------------------------------------------
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType type, uint64_t inner,
                         uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle swizzle) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  TmapKey key{dev, base, static_cast<int>(type), inner, outer, row_bytes, box_inner, box_outer,
              static_cast<int>(swizzle)};
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& t : g_tmaps) {
    if (t.used && t.key == key) {
      t.stamp = ++g_tmap_clock;
      *map = t.map;
      return cudaSuccess;
    }
  }
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
      t_fail_site = GP_SITE_TENSOR_MAP;
      return e != cudaSuccess ? e : cudaErrorNotSupported;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // The encode is a driver call: it needs the device's context current in this
  // host thread, which a thread that has only queried the device may not have
  // yet (cudaSetDevice makes the primary context current).
  thread_local int ctx_dev = -1;
  if (ctx_dev != dev) {
    if ((e = cudaSetDevice(dev)) != cudaSuccess) {
      t_fail_site = GP_SITE_TENSOR_MAP;
      return e;
    }
    ctx_dev = dev;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  const CUresult r = g_encode(&m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_fail_site = GP_SITE_TENSOR_MAP;
    return cudaErrorInvalidValue;
  }
  TmapEntry* victim = &g_tmaps[0];
  for (auto& t : g_tmaps) {
    if (!t.used) { victim = &t; break; }
    if (t.stamp < victim->stamp) victim = &t;
  }
  victim->key = key;
  victim->map = m;
  victim->stamp = ++g_tmap_clock;
  victim->used = true;
  *map = m;
  return cudaSuccess;
}

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (done.count({dev, kernel})) return cudaSuccess;
  }
  // the opt-in limit covers static and dynamic shared memory together
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  const int max_dynamic = kSmemPerCtaMax - static_cast<int>(fa.sharedSizeBytes);
  if (e == cudaSuccess && bytes > max_dynamic) e = cudaErrorInvalidValue;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic);
  if (e != cudaSuccess) {
    t_fail_site = GP_SITE_SMEM_ATTR;
    return e;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  done.insert({dev, kernel});
  return cudaSuccess;
}

namespace {
__global__ void zero_fill_kernel(uint4* p, int64_t n16) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0, 0, 0, 0);
}
}  // namespace

cudaError_t launch_zero_fill(void* C, int64_t bytes, cudaStream_t stream) {
  const int64_t n16 = bytes / 16;   // output rows are multiples of 16 bytes under the alignment rules
  if (n16 <= 0) return cudaSuccess;
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  zero_fill_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(static_cast<uint4*>(C), n16);
  return cudaGetLastError();
}

}  // namespace gp

namespace gp {
// ---------------------------------------------------------------------------
// allocation-free entry point (gemm_pipelined_noalloc): fixed scratch array
// ---------------------------------------------------------------------------
// Stream-K scratch of gemm_pipelined_noalloc: FP32 partial tiles followed by
// the split-tile counters.  It is a static device array, so every GPU that
// loads this library holds it (41 MiB + 64 KiB) until the process exits, and
// no call ever allocates.  40 MiB of partials covers every split plan of the
// FP16/BF16 ring on a 152-SM GB300 (152 CTAs x 2 slots x 128 x 256 x 4 B).
constexpr size_t kNoAllocPartialBytes = size_t(40) << 20;
constexpr size_t kNoAllocCounterBytes = size_t(64) << 10;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocPartialBytes + kNoAllocCounterBytes];

namespace {
struct NoAllocDevice {
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  uint32_t epoch = 0;                 // tag of the counts of the latest call on this device
};
NoAllocDevice g_noalloc[kMaxDevices];

// Once per device, with that device current: translate the array's host-side
// name into its device address and zero the counters.  Returns the address
// and the epoch for this call.
cudaError_t noalloc_setup(int dev, unsigned char** scratch, uint32_t* epoch) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.scratch) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemset(static_cast<unsigned char*>(p) + kNoAllocPartialBytes, 0, kNoAllocCounterBytes);
    if (e != cudaSuccess) return e;
    d.scratch = static_cast<unsigned char*>(p);
  }
  if (++d.epoch == 0) d.epoch = 1;
  *scratch = d.scratch;
  *epoch = d.epoch;
  return cudaSuccess;
}
}  // namespace
}  // namespace gp

using namespace gp;

extern "C" {

int gemm_abi_version(void) { return 10700; }

const char* gemm_strerror(int code) {
  switch (code) {
    case GP_OK: return "ok";
    case GP_ERR_ARG: return "invalid argument";
    case GP_ERR_UNSUPPORTED: return "unsupported dtype/layout/variant combination or alignment";
    case GP_ERR_SMEM: return "no tile fits the shared-memory budget at this stage count";
    case GP_ERR_CUDA: return "CUDA runtime or launch error";
    case GP_ERR_TIMEOUT: return "a bounded wait inside the kernel timed out";
    case GP_ERR_SIZE: return "a dimension is too large for this kernel";
    case GP_ERR_SCRATCH: return "the plan needs more scratch memory than the fixed device array holds";
    default: return "unknown error code";
  }
}

int gemm_plan(int64_t M, int64_t N, int64_t K, int dtype, int layout, int stages, int variant, int bn,
              gp_plan* out) {
  if (!out) return GP_ERR_ARG;
  int sms = 0;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  } else {
    cudaGetLastError();   // clear the sticky "no device" error of the probe
  }
  return plan_impl(M, N, K, dtype, layout, stages, variant, bn, sms, out);
}

int gemm_plan_ex(int64_t M, int64_t N, int64_t K, int dtype, int layout, int stages, int variant,
                 const gp_options* opts, gp_plan* out) {
  if (!out) return GP_ERR_ARG;
  if (opts && opts->plan_sms < 0) return GP_ERR_ARG;
  int sms = 0;
  int ndev = 0;
  if (opts && opts->plan_sms > 0) {
    sms = opts->plan_sms;
  } else if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  } else {
    cudaGetLastError();
  }
  const bool no_pair = opts && (opts->no_cta_pair || opts->inject_lost_load);
  return plan_impl(M, N, K, dtype, layout, stages, variant, opts ? opts->bn : 0, sms, out, opts && opts->no_stream_k,
                   no_pair, opts ? opts->i8_engine : 0, opts ? opts->ffma_tm : 0, opts ? opts->ffma_tn : 0,
                   opts ? opts->pair_k_split : 0, opts && opts->one_tile_per_cta, opts ? opts->raster_gm : 0);
}

int gemm_pipelined_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype, int layout,
                      int stages, int variant, void* stream, const gp_options* opts) {
  std::memset(&t_last.stats, 0, sizeof(t_last.stats));
  t_last.status_slot = nullptr;
  t_last.call_id = 0;
  t_fail_site = 0;
  t_last.stats.last_ms = -1.f;
  t_last.kernel = nullptr;
  t_last.timed = false;
  t_last.stream = static_cast<cudaStream_t>(stream);
  const int bn_req = opts ? opts->bn : 0;

  // argument checks that need no device
  gp_plan plan;
  int rc = plan_impl(M, N, K, dtype, layout, stages, variant, bn_req, 0, &plan, opts && opts->no_stream_k,
                     opts && (opts->no_cta_pair || opts->inject_lost_load), opts ? opts->i8_engine : 0,
                     opts ? opts->ffma_tm : 0, opts ? opts->ffma_tn : 0, opts ? opts->pair_k_split : 0,
                     opts && opts->one_tile_per_cta, opts ? opts->raster_gm : 0);
  if (rc != GP_OK) { record(rc, 0); return rc; }
  t_last.stats.plan = plan;
  if (M == 0 || N == 0) { record(GP_OK, 0); return GP_OK; }   // empty output: nothing read or written
  if (!C || (K > 0 && (!A || !B))) {
    record(GP_ERR_ARG, 0);
    return GP_ERR_ARG;
  }
  if (!alignment_ok(A, B, C, N, K, dtype)) { record(GP_ERR_UNSUPPORTED, 0); return GP_ERR_UNSUPPORTED; }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  unsigned long long* status = nullptr;
  uint32_t call_id = 0;
  int sms = 0;
  if (e == cudaSuccess) e = device_info(dev, &sms, &call_id, &status);
  if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_DEVICE); return GP_ERR_CUDA; }
  t_last.device = dev;
  t_last.status_slot = status;
  t_last.call_id = call_id;
  t_last.stats.sm_count = sms;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool timed = opts && opts->time_kernel;
  if (timed) {
    if (t_last.ev_device != dev) {
      if (t_last.ev[0]) { cudaEventDestroy(t_last.ev[0]); cudaEventDestroy(t_last.ev[1]); }
      t_last.ev[0] = t_last.ev[1] = nullptr;
      if ((e = cudaEventCreate(&t_last.ev[0])) != cudaSuccess || (e = cudaEventCreate(&t_last.ev[1])) != cudaSuccess) {
        record(GP_ERR_CUDA, e, GP_SITE_EVENT);
        return GP_ERR_CUDA;
      }
      t_last.ev_device = dev;
    }
    cudaEventRecord(t_last.ev[0], st);
  }

  if (K == 0) {
    e = launch_zero_fill(C, M * N * out_elem_bytes(dtype), st);
  } else {
    const bool no_pair = opts && (opts->no_cta_pair || opts->inject_lost_load);
    rc = plan_impl(M, N, K, dtype, layout, stages, variant, bn_req, sms, &plan, opts && opts->no_stream_k, no_pair,
                   opts ? opts->i8_engine : 0, opts ? opts->ffma_tm : 0, opts ? opts->ffma_tn : 0,
                   opts ? opts->pair_k_split : 0, opts && opts->one_tile_per_cta, opts ? opts->raster_gm : 0);
    if (rc != GP_OK) { record(rc, 0); return rc; }
    if (plan.cta_pair == 3) {
      int clusters = 0;
      e = umma_kx_capacity(dtype, plan.smem_bytes, &clusters);
      if (e == cudaSuccess && clusters < 1) e = cudaErrorLaunchOutOfResources;
      if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_CAPACITY); return GP_ERR_CUDA; }
      if (4 * clusters < plan.grid) plan.grid = 4 * clusters;
    }
    void* conv = nullptr;
    const bool i8_overlap = plan.cta_pair && dtype == GP_I8_I32 && plan.kernel == kI8OverlapKernelName;
    const bool i8_tc = plan.cta_pair && dtype == GP_I8_I32;   // both engines keep FP16 copies
    const int64_t conv_bytes = i8_tc ? i8_conv_bytes(M, N, K) : 0;
    uint32_t* conv_ctrs = nullptr;
    int32_t conv_kcap = 0;
    uint32_t conv_parity = 0;
    if (plan.cta_pair == 1) {
      // pairs must sit on one TPC each: the resident count may be below SMs / 2
      int pairs = 0;
      e = umma_pair_capacity(dtype, plan.smem_bytes, &pairs, i8_overlap);
      if (e == cudaSuccess && pairs < 1) e = cudaErrorLaunchOutOfResources;
      if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_CAPACITY); return GP_ERR_CUDA; }
      if (pairs < sms / 2 && !i8_overlap && (!i8_tc || plan.tiles < pairs)) {
        apply_stream_k(&plan, pairs, 2, !(opts && opts->no_stream_k));
        plan.workspace_bytes += conv_bytes;
      }
      if (i8_tc && !i8_overlap) apply_i8_halves(&plan, pairs);
      if (i8_tc) {
        e = get_conv_workspace(dev, st, static_cast<size_t>(conv_bytes), &conv,
                               !i8_overlap && opts && opts->inputs_ready);
        if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_WORKSPACE); return GP_ERR_CUDA; }
      }
      if (i8_overlap) {
        e = get_overlap_ctrs(dev, st, plan.k_tiles, &conv_ctrs, &conv_kcap, &conv_parity);
        if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_WORKSPACE); return GP_ERR_CUDA; }
      }
    }
    SkParams sk{plan.dp_tiles, plan.sk_tiles, nullptr, nullptr, 0, plan.raster_gm, plan.b_resident};
    if (plan.sk_tiles > 0) {
      const size_t counter_words =
          static_cast<size_t>(plan.sk_tiles) * (plan.cta_pair ? 2 : 1) * 2;
      e = get_workspace(dev, st, static_cast<size_t>(plan.workspace_bytes - conv_bytes), counter_words, &sk.workspace,
                        &sk.flags, &sk.epoch);
      if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_WORKSPACE); return GP_ERR_CUDA; }
    }
    FfmaSplit ks{plan.k_splits, nullptr, nullptr, 0};
    if (plan.k_splits > 1) {
      uint32_t* counters = nullptr;
      e = get_workspace(dev, st, static_cast<size_t>(plan.workspace_bytes), static_cast<size_t>(plan.tiles) * 2,
                        &ks.workspace, &counters, &ks.epoch);
      if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_WORKSPACE); return GP_ERR_CUDA; }
      ks.counters = reinterpret_cast<unsigned long long*>(counters);
    }
    LaunchArgs a;
    a.A = A;
    a.B = B;
    a.C = C;
    a.M = static_cast<int32_t>(M);
    a.N = static_cast<int32_t>(N);
    a.K = static_cast<int32_t>(K);
    a.dtype = dtype;
    a.layout = layout;
    a.variant = variant;
    a.plan = plan;
    a.stream = st;
    a.ctl.status = status;
    a.ctl.call_id = call_id;
    a.ctl.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : kDefaultTimeoutNs;
    a.ctl.inject_lost_load = opts ? opts->inject_lost_load : 0;
    a.ctl.inputs_ready = (opts && opts->inputs_ready) ? 1 : 0;
    a.sm_count = sms;
    a.sk = sk;
    a.ks = ks;
    a.ffma_tm = (opts && opts->ffma_tm) ? opts->ffma_tm : 8;
    a.ffma_tn = (opts && opts->ffma_tn) ? opts->ffma_tn : 8;
    a.conv = conv;
    a.i8_overlap = i8_overlap;
    a.conv_early = !i8_overlap && opts && opts->inputs_ready;
    a.conv_ctrs = conv_ctrs;
    a.conv_kcap = conv_kcap;
    a.conv_parity = conv_parity;
    a.one_tile = opts && opts->one_tile_per_cta;
    const void* kernel = nullptr;
    switch (family_of(dtype)) {
      case 0: e = launch_ffma(a, &kernel); break;
      case 1: e = plan.cta_pair ? launch_umma_i8(a, &kernel) : launch_imma(a, &kernel); break;
      default: e = launch_umma(a, &kernel); break;
    }
    // A launch that did not start left its successor's counter set unzeroed: clear both sets.
    if (e != cudaSuccess && i8_overlap)
      cudaMemsetAsync(conv_ctrs, 0, 2 * static_cast<size_t>(conv_kcap + 1) * sizeof(uint32_t), st);
    t_last.stats.plan = a.plan;
    t_last.kernel = kernel;
  }
  if (e != cudaSuccess) {
    record(GP_ERR_CUDA, e, t_fail_site ? t_fail_site : GP_SITE_LAUNCH);
    return GP_ERR_CUDA;
  }
  if (timed) {
    cudaEventRecord(t_last.ev[1], st);
    t_last.timed = true;
  }
  record(GP_OK, 0);
  return GP_OK;
}

int gemm_release(int device) {
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
    cudaGetLastError();
    return GP_ERR_CUDA;
  }
  if (device < 0 || device >= ndev || device >= kMaxDevices) return GP_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = 0;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return GP_ERR_CUDA;
  if (cur != device && (e = cudaSetDevice(device)) != cudaSuccess) return GP_ERR_CUDA;
  e = cudaDeviceSynchronize();   // nothing on any stream of the device still uses a workspace
  if (e == cudaSuccess)
    for (auto& w : g_ws)
      if (w.dev == device) free_workspace(w);
  if (cur != device) cudaSetDevice(cur);
  return e == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

int gemm_pipelined(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype, int layout,
                   int stages, int variant, void* stream) {
  return gemm_pipelined_ex(A, B, C, M, N, K, dtype, layout, stages, variant, stream, nullptr);
}

int gemm_stats(gp_stats* out, int sync) {
  if (!out) return GP_ERR_ARG;
  if (!t_last.valid) {
    std::memset(out, 0, sizeof(*out));
    out->last_ms = -1.f;
    return GP_OK;
  }
  gp_stats& s = t_last.stats;
  if (sync && t_last.device >= 0 && s.status == GP_OK) {
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != t_last.device) cudaSetDevice(t_last.device);
    // the call's status slot, read on the call's own stream (after the call)
    unsigned long long word = 0;
    cudaError_t e = cudaSuccess;
    if (t_last.status_slot)
      e = cudaMemcpyAsync(&word, t_last.status_slot, sizeof(word), cudaMemcpyDeviceToHost, t_last.stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(t_last.stream);
    if (e == cudaSuccess && t_last.status_slot && static_cast<uint32_t>(word >> 32) == t_last.call_id &&
        static_cast<uint32_t>(word) != 0) {
      s.device_status = static_cast<uint32_t>(word);
      s.status = GP_ERR_TIMEOUT;
    }
    if (e != cudaSuccess) {
      s.status = GP_ERR_CUDA;
      s.cuda_error = e;
      s.cuda_error_site = GP_SITE_SYNC;
    } else if (t_last.timed) {
      float ms = -1.f;
      if (cudaEventElapsedTime(&ms, t_last.ev[0], t_last.ev[1]) == cudaSuccess) s.last_ms = ms;
      t_last.timed = false;
    }
    if (prev != t_last.device) cudaSetDevice(prev);
  }
  if (t_last.kernel && s.regs_per_thread == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, t_last.kernel) == cudaSuccess) {
      s.regs_per_thread = fa.numRegs;
      s.local_bytes = static_cast<int32_t>(fa.localSizeBytes);
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, t_last.kernel, s.plan.threads, s.plan.smem_bytes) ==
        cudaSuccess)
      s.blocks_per_sm = occ;
  }
  *out = s;
  return s.status;
}

int gemm_pipelined_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype,
                           int stages, void* stream) {
  std::memset(&t_last.stats, 0, sizeof(t_last.stats));
  t_last.status_slot = nullptr;
  t_last.call_id = 0;
  t_fail_site = 0;
  t_last.stats.last_ms = -1.f;
  t_last.kernel = nullptr;
  t_last.timed = false;
  t_last.stream = static_cast<cudaStream_t>(stream);
  if (dtype != GP_F16_F32ACC_F16OUT && dtype != GP_BF16_F32ACC_BF16OUT) {
    record(GP_ERR_UNSUPPORTED, 0);
    return GP_ERR_UNSUPPORTED;
  }
  gp_plan plan;
  // (plain CTA pairs: the fixed scratch is sized for them)
  int rc = plan_impl(M, N, K, dtype, GP_A_ROW_B_COL, stages, GP_PIPELINED, 0, 0, &plan, false, false, 0, 0, 0, 0);
  if (rc != GP_OK) { record(rc, 0); return rc; }
  t_last.stats.plan = plan;
  if (M == 0 || N == 0) { record(GP_OK, 0); return GP_OK; }
  if (!C || (K > 0 && (!A || !B))) { record(GP_ERR_ARG, 0); return GP_ERR_ARG; }
  if (!alignment_ok(A, B, C, N, K, dtype)) { record(GP_ERR_UNSUPPORTED, 0); return GP_ERR_UNSUPPORTED; }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  unsigned long long* status = nullptr;
  uint32_t call_id = 0;
  int sms = 0;
  if (e == cudaSuccess) e = device_info(dev, &sms, &call_id, &status);
  unsigned char* scratch = nullptr;
  uint32_t epoch = 0;
  if (e == cudaSuccess) e = noalloc_setup(dev, &scratch, &epoch);
  if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_DEVICE); return GP_ERR_CUDA; }
  t_last.device = dev;
  t_last.status_slot = status;
  t_last.call_id = call_id;
  t_last.stats.sm_count = sms;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (K == 0) {
    e = launch_zero_fill(C, M * N * out_elem_bytes(dtype), st);
  } else {
    rc = plan_impl(M, N, K, dtype, GP_A_ROW_B_COL, stages, GP_PIPELINED, 0, sms, &plan, false, false, 0, 0, 0, 0);
    if (rc != GP_OK) { record(rc, 0); return rc; }
    if (plan.cta_pair) {
      int pairs = 0;
      e = umma_pair_capacity(dtype, plan.smem_bytes, &pairs);
      if (e == cudaSuccess && pairs < 1) e = cudaErrorLaunchOutOfResources;
      if (e != cudaSuccess) { record(GP_ERR_CUDA, e, GP_SITE_CAPACITY); return GP_ERR_CUDA; }
      if (pairs < sms / 2) apply_stream_k(&plan, pairs, 2, true);
    }
    t_last.stats.plan = plan;
    SkParams sk{plan.dp_tiles, plan.sk_tiles, nullptr, nullptr, epoch, plan.raster_gm, plan.b_resident};
    if (plan.sk_tiles > 0) {
      const size_t counter_bytes = static_cast<size_t>(plan.sk_tiles) * (plan.cta_pair ? 2 : 1) * 8;
      if (static_cast<size_t>(plan.workspace_bytes) > kNoAllocPartialBytes || counter_bytes > kNoAllocCounterBytes) {
        record(GP_ERR_SCRATCH, 0);
        return GP_ERR_SCRATCH;
      }
      sk.workspace = reinterpret_cast<float*>(scratch);
      sk.flags = reinterpret_cast<uint32_t*>(scratch + kNoAllocPartialBytes);
    }
    LaunchArgs a;
    a.A = A;
    a.B = B;
    a.C = C;
    a.M = static_cast<int32_t>(M);
    a.N = static_cast<int32_t>(N);
    a.K = static_cast<int32_t>(K);
    a.dtype = dtype;
    a.layout = GP_A_ROW_B_COL;
    a.variant = GP_PIPELINED;
    a.plan = plan;
    a.stream = st;
    a.ctl.status = status;
    a.ctl.call_id = call_id;
    a.ctl.timeout_ns = kDefaultTimeoutNs;
    a.ctl.inject_lost_load = 0;
    a.ctl.inputs_ready = 0;
    a.sm_count = sms;
    a.sk = sk;
    a.ks = FfmaSplit{1, nullptr, nullptr, 0};
    a.ffma_tm = a.ffma_tn = 8;
    a.conv = nullptr;
    a.i8_overlap = false;
    a.conv_early = false;
    a.conv_ctrs = nullptr;
    a.conv_kcap = 0;
    a.conv_parity = 0;
    a.one_tile = false;
    const void* kernel = nullptr;
    e = launch_umma(a, &kernel);
    t_last.stats.plan = a.plan;
    t_last.kernel = kernel;
  }
  if (e != cudaSuccess) {
    record(GP_ERR_CUDA, e, t_fail_site ? t_fail_site : GP_SITE_LAUNCH);
    return GP_ERR_CUDA;
  }
  record(GP_OK, 0);
  return GP_OK;
}

}  // extern "C"
