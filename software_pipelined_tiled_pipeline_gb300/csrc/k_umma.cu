// k_umma.cu -- FP16/BF16 GEMM on the 5th-generation tensor cores (tcgen05.mma,
// FP32 accumulators in TMEM), three data paths for the K-loop:
//
//  * umma_ring_kernel  -- the main path.  Persistent, warp-specialised:
//      warp 0  TMA producer: fills an S-slot shared-memory ring, one slot per
//              K step, guarded by mbarrier full/empty phases;
//      warp 1  allocates TMEM and issues tcgen05.mma (one thread), releasing
//              each slot with tcgen05.commit -> empty[s];
//      warps 2-5 epilogue: TMEM -> registers (tcgen05.ld) -> FP16/BF16 ->
//              swizzled shared staging -> TMA store.
//    The accumulator is double-buffered in TMEM so the epilogue of one tile
//    overlaps the K-loop of the next.  When the output tiles do not divide
//    evenly over the CTAs, the K-loops of the last ones are split evenly
//    across all CTAs (stream-K): each segment stores an FP32 partial in a
//    workspace and the segment that completes last sums them and writes C,
//    so no CTA ever waits on another.  This is the S-stage ring of
//    "CUDA Kernel Study: Pipelining", Case 2 (prologue fills S slots, the
//    steady state refills the slot just consumed, the tail drains), with TMA
//    completion bytes on an mbarrier in place of cp.async commit/wait groups.
//
//  * umma_staged_kernel<PINGPONG=true> -- the register-staged double buffer of Case 1 /
//    "pipeline-gpu-kernel" Step 3 (LDG-register variant): global loads of tile
//    k+1 into registers are in flight while the tensor core consumes tile k
//    from one shared buffer; the registers are then stored to the other
//    buffer.  The "compute finished reading" barrier before that store is the
//    tcgen05.commit of the previous tile's MMAs.
//
//  * umma_staged_kernel<PINGPONG=false> -- load, synchronise, compute, wait (Background).
//
// All three use the same tile shape, shared-memory layout (K-major tiles of
// 128-byte rows with the 128-byte swizzle), MMA sequence and epilogue, so
// they differ only in how tiles reach shared memory.
#include <atomic>
#include "gp_device.cuh"

namespace gp {
namespace {

constexpr int BM = kUmmaBM;   // 128
constexpr int BK = kUmmaBK;   // 64 elements = 128 bytes per row
constexpr int A_BYTES = BM * BK * 2;
constexpr int UMMA_K = 16;    // K of one kind::f16 instruction
constexpr uint64_t kSkPollNs = 20000;   // how long a split tile's first-K-step owner polls for the others

struct UmmaBarriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done[2];
  uint64_t drain;
  uint64_t xfull, xempty;     // K split over two pairs: the other pair's accumulator half is in xbuf / xbuf is free
  uint32_t tmem_base;
  int32_t consumed_hi;        // k-blocks consumed by the MMA thread (low 31 bits)
  CtaCtl ctl;
  int32_t sk_last;            // epilogue: this CTA completed the last segment of a split tile
};
static_assert(sizeof(UmmaBarriers) <= kBarrierRegion, "barrier region too small");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Grouped raster: GM consecutive M-blocks share each N-block sweep, so the
// CTAs resident at one time reuse A and B tiles through L2 (GM = 8 for the
// one-tile-per-CTA kernels; the persistent rings take it from the plan).
constexpr int kRasterGM = 8;
__device__ __forceinline__ void tile_coords(int tile, int m_blocks, int n_blocks, int& mb, int& nb,
                                            int GM = kRasterGM) {
  const int per_group = GM * n_blocks;
  const int group = tile / per_group;
  const int first_m = group * GM;
  const int gm = min(GM, m_blocks - first_m);
  const int in_group = tile - group * per_group;
  mb = first_m + in_group % gm;
  nb = in_group / gm;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Store one 32-row x 64-column chunk of the accumulator (already in registers,
// FP32 bit patterns) to C through a 4 KB swizzled staging buffer and a TMA
// store.  Lane t holds row (row0 + t).  The caller guarantees the staging
// buffer is free (no TMA store still reading it).
template <bool BF16>
__device__ __forceinline__ void pack_chunk(const uint32_t (&v)[64], uint32_t (&p)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) p[i] = pack2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), BF16);
}

// Stage one packed 32-row x 64-column chunk (lane t: row t, 128 bytes) and store it with TMA.
__device__ __forceinline__ void store_packed(const uint32_t (&p)[32], uint8_t* buf, int lane,
                                             const CUtensorMap* tmap_c, int x, int y, bool in_bounds) {
  const uint32_t base = smem_u32(buf);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t addr = base + sw128_offset(lane, j);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(p[4 * j]), "r"(p[4 * j + 1]),
                 "r"(p[4 * j + 2]), "r"(p[4 * j + 3])
                 : "memory");
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && in_bounds) tma_store_2d(tmap_c, base, x, y);
  if (lane == 0) bulk_commit();
}

template <bool BF16>
__device__ __forceinline__ void stage_and_store(const uint32_t (&v)[64], uint8_t* buf, int lane,
                                                const CUtensorMap* tmap_c, int x, int y, bool in_bounds) {
  uint32_t p[32];
  pack_chunk<BF16>(v, p);
  store_packed(p, buf, lane, tmap_c, x, y, in_bounds);
}

// Start reading 64 accumulator columns of this warp's 32 TMEM lanes into v;
// v is valid after tmem_wait_ld().
__device__ __forceinline__ void issue_acc_chunk(uint32_t taddr, uint32_t (&v)[64]) {
  uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
  uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
  tmem_ld_32x32b_x32(taddr, lo);
  tmem_ld_32x32b_x32(taddr + 32, hi);
}

__device__ __forceinline__ void load_acc_chunk(uint32_t taddr, uint32_t (&v)[64]) {
  issue_acc_chunk(taddr, v);
  tmem_wait_ld();
  regs_after_wait(v);
}

// Issue the four K=16 UMMAs of one 64-wide K step from slot (a_addr, b_addr).
template <int BN>
__device__ __forceinline__ void umma_kblock(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, uint32_t idesc,
                                            bool first) {
  const uint64_t da = umma_desc_sw128(a_addr);
  const uint64_t db = umma_desc_sw128(b_addr);
#pragma unroll
  for (int kk = 0; kk < BK / UMMA_K; ++kk) {
    // advancing the start address by 32 bytes (>> 4 = 2) steps 16 elements along K
    umma_f16(d_tmem, da + 2 * kk, db + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
  }
}

// ---------------------------------------------------------------------------
// main path: persistent warp-specialised TMA ring
// ---------------------------------------------------------------------------

// The ordered list of work items of one worker (a CTA, or a CTA pair), walked
// identically by the producer, the MMA issuer and the epilogue: its first
// whole tile (w), then its contiguous range of the stream-K units (one unit =
// one K step of one of the sk_tiles tiles after the whole ones), cut at tile
// boundaries, then its other whole tiles (w+W, w+2W, ... below dp_tiles).
// (The split tiles are those left after the full waves, or after all but the
// last full wave with a shallow ring: the planner decides.)
// The split tiles come before the last whole tiles so that their partial-tile
// traffic and fix-ups overlap MMAs instead of trailing the kernel (measured:
// the fix-up of a split tile takes 6-8 us after its last MMA); one whole tile
// goes first because all workers then start on neighbouring tiles at K step
// 0, whose operands they share in L2 (measured +2 % at 4096^3).  An item is
// (tile, first K step, one past the last K step).  With B kept in the ring
// (SkParams.b_resident) a worker instead walks one contiguous run of whole
// tiles, so that consecutive tiles share their N block.
struct WorkIter {
  int dp_tiles, kt, next_dp, step;
  int64_t u, u_end;
  bool first_done;

  __device__ __forceinline__ static int64_t range_start(int w, int64_t units, int workers) {
    return static_cast<int64_t>(w) * units / workers;
  }
  __device__ __forceinline__ void init(const SkParams& sk, int kt_, int worker, int workers) {
    kt = kt_;
    first_done = false;
    if (sk.b_resident) {
      // whole tiles only: worker w takes the contiguous run [w T / W, (w + 1) T / W)
      next_dp = static_cast<int>(range_start(worker, sk.dp_tiles, workers));
      dp_tiles = static_cast<int>(range_start(worker + 1, sk.dp_tiles, workers));
      step = 1;
      u = u_end = 0;
      return;
    }
    dp_tiles = sk.dp_tiles;
    next_dp = worker;
    step = workers;
    const int64_t units = static_cast<int64_t>(sk.sk_tiles) * kt;
    u = range_start(worker, units, workers);
    u_end = range_start(worker + 1, units, workers);
  }
  __device__ __forceinline__ bool next(int& tile, int& k0, int& k1) {
    if (!first_done) {
      first_done = true;
      if (next_dp < dp_tiles) {
        tile = next_dp;
        k0 = 0;
        k1 = kt;
        next_dp += step;
        return true;
      }
    }
    if (u < u_end) {
      const int t = static_cast<int>(u / kt);
      k0 = static_cast<int>(u - static_cast<int64_t>(t) * kt);
      const int64_t left = u_end - u;
      k1 = (left < kt - k0) ? k0 + static_cast<int>(left) : kt;
      tile = dp_tiles + t;
      u += k1 - k0;
      return true;
    }
    if (next_dp < dp_tiles) {
      tile = next_dp;
      k0 = 0;
      k1 = kt;
      next_dp += step;
      return true;
    }
    return false;
  }
};

// One tile of the stream-K range as the epilogue sees it: the workers whose
// unit ranges overlap its K steps (w_first .. w_last; a worker whose range is
// empty holds no segment), the number of segments, and the tile's 64-bit
// counter {launch epoch, segments counted} for this CTA rank.
struct SplitTile {
  int64_t start;     // stream-K unit of the tile's first K step
  int64_t units;     // units of the whole stream-K range
  int workers;
  int w_first, w_last, segments;
  unsigned long long* ctr;

  __device__ __forceinline__ void init(int tile, int kt, const SkParams& sk, int workers_, int ctas, uint32_t rank) {
    workers = workers_;
    units = static_cast<int64_t>(sk.sk_tiles) * kt;
    start = static_cast<int64_t>(tile - sk.dp_tiles) * kt;
    const int64_t end = start + kt;
    w_first = static_cast<int>(start * workers / units);
    while (w_first + 1 < workers && WorkIter::range_start(w_first + 1, units, workers) <= start) ++w_first;
    while (w_first > 0 && WorkIter::range_start(w_first, units, workers) > start) --w_first;
    w_last = w_first;
    while (w_last + 1 < workers && WorkIter::range_start(w_last + 1, units, workers) < end) ++w_last;
    segments = 0;
    for (int w = w_first; w <= w_last; ++w) segments += has_segment(w);
    ctr = reinterpret_cast<unsigned long long*>(sk.flags) + static_cast<int64_t>(tile - sk.dp_tiles) * ctas + rank;
  }
  __device__ __forceinline__ bool has_segment(int w) const {
    return WorkIter::range_start(w, units, workers) < WorkIter::range_start(w + 1, units, workers);
  }
  // Workspace slot of worker w's segment of this tile: (2w + j) * CTAs + rank,
  // j = 0 if it is the worker's first segment, 1 if its last.
  __device__ __forceinline__ int slot(int w, int ctas, uint32_t rank) const {
    return (2 * w + (WorkIter::range_start(w, units, workers) >= start ? 0 : 1)) * ctas + static_cast<int>(rank);
  }
  __device__ __forceinline__ static uint32_t count_of(unsigned long long word, uint32_t epoch) {
    return (static_cast<uint32_t>(word >> 32) == epoch) ? static_cast<uint32_t>(word) : 0u;
  }
  // The owner of the first K step: true if every other segment is counted
  // within kSkPollNs (bounded; false means fall back to counting in).
  __device__ __forceinline__ bool poll_others(uint32_t epoch) const {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
      if (count_of(*reinterpret_cast<volatile unsigned long long*>(ctr), epoch) + 1u ==
          static_cast<uint32_t>(segments))
        return true;
      if (global_timer_ns() - t0 > kSkPollNs) return false;
      __nanosleep(128);
    }
  }
  // Count this segment in; true if it was the last one of the tile.
  __device__ __forceinline__ bool count_in(uint32_t epoch) const {
    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr);
    for (;;) {
      const uint32_t count = count_of(old, epoch);
      const unsigned long long want = (static_cast<unsigned long long>(epoch) << 32) | (count + 1u);
      const unsigned long long seen = atomicCAS(ctr, old, want);
      if (seen == old) return count + 1u == static_cast<uint32_t>(segments);
      old = seen;
    }
  }
};

// Partial tiles are stored column-quad-major, row innermost: 16-byte group i
// (4 columns) of 64-column chunk c of row r in slot p at
// ((p * BN/64 + c) * 16 + i) * 128 + r, so the 32 lanes of a warp (32
// consecutive rows) touch 512 contiguous bytes.  Index in 16-byte units.
template <int BN>
__device__ __forceinline__ size_t partial_at(int slot, int c, int i, int row) {
  return ((static_cast<size_t>(slot) * (BN / kUmmaEpiCols) + c) * 16 + i) * 128 + row;
}

template <int THREADS>
__device__ __forceinline__ void epi_bar_sync() {   // the epilogue warps only
  asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
}

// Barrier of the epilogue warps that also ANDs a predicate over their threads.
template <int THREADS>
__device__ __forceinline__ bool epi_bar_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "n"(THREADS)
      : "memory");
  return r != 0;
}

// Shapes of the ring kernel.  PAIR = false: one CTA per 128 x BN tile.
// PAIR = true (BN = 256): a cluster of two CTAs per 256 x 256 tile; each CTA
// loads its own 128-row halves of the A and B tiles (32 KB per K step instead
// of the 48 KB one CTA needs for 128 x 256), one thread of the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256), which reads both CTAs' halves and writes
// each CTA's 128 accumulator rows into that CTA's TMEM.  The even CTA's
// full[s] barrier counts the bytes of both CTAs' loads (the odd CTA's TMA
// signals it through the cluster window); the MMA commit releases slot s in
// both CTAs at once, so the two producers run in lockstep; epilogue warps of
// both CTAs hand an accumulator back by arriving on the even CTA's acc_empty.
// Epilogue: warp w may read TMEM lanes 32 (w mod 4) .. +31 only, so four warps
// cover the 128 rows, each taking every 64-column chunk of its rows.  (The
// code also runs with eight, two per lane quarter splitting the columns; at
// 10 warps a thread gets at most 168 registers, and the measured epilogue was
// no faster, so the kernel uses four.)
template <int BN, bool PAIR>
struct RingShape {
  static constexpr int A_ROWS = 128;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;
  static constexpr int A_BYTES = A_ROWS * BK * 2;
  static constexpr int STAGE = (A_ROWS + B_ROWS) * BK * 2;
  static constexpr int TILE_M = PAIR ? 2 * A_ROWS : A_ROWS;
  static constexpr int CTAS = PAIR ? 2 : 1;
  static constexpr uint32_t TMEM_COLS = 2 * BN;   // double-buffered 128 x BN FP32 accumulator per CTA
  static constexpr int EPI_WARPS = 4;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 64 + EPI_THREADS;
  static constexpr int CHUNKS = BN / kUmmaEpiCols;                 // 64-column chunks per accumulator row
  static constexpr int WARP_CHUNKS = CHUNKS / (EPI_WARPS / 4);     // chunks per epilogue warp
  static constexpr int EPI_BUFS = kUmmaEpiBytes / (EPI_WARPS * kUmmaEpiBufBytes);   // staging buffers per warp
  static_assert(EPI_BUFS >= 1 && WARP_CHUNKS >= 1, "epilogue split");
};

template <int BN, bool BF16, bool PAIR, bool KX>
__global__ void __launch_bounds__(RingShape<BN, PAIR>::THREADS, 1)
    umma_ring_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, int M, int N, int K, int stages, KernelCtl ctl,
                     SkParams sk) {
  using Sh = RingShape<BN, PAIR>;
  constexpr int STAGE = Sh::STAGE;
  constexpr uint32_t IDESC = umma_idesc_f16(BF16, Sh::TILE_M, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* epi = smem + stages * STAGE;
  UmmaBarriers* bar = reinterpret_cast<UmmaBarriers*>(epi + kUmmaEpiBytes);
  float4* xbuf = reinterpret_cast<float4*>(epi + kUmmaEpiBytes + kBarrierRegion);   // KX only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // KX: a cluster of two CTA pairs computes one 256 x BN tile, pair p the
  // K steps p*ceil(kt/2) .. of it; pair 1 sends its FP32 accumulator through
  // distributed shared memory to pair 0, which adds it and writes C.
  constexpr int CL = KX ? 4 : (PAIR ? 2 : 1);                 // CTAs per worker (one cluster)
  static_assert(!KX || (PAIR && BN == 128), "K split runs on 256 x 128 pair tiles");
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;      // rank in the cluster
  const uint32_t rank = crank & 1u;                           // rank in the CTA pair
  const int pidx = KX ? static_cast<int>(crank >> 1) : 0;   // pair within the cluster
  const bool leader = rank == 0;
  const uint32_t lead_rank = crank & ~1u;                     // this pair's even CTA
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << lead_rank);
  const int worker = static_cast<int>(blockIdx.x) / CL;
  const int workers = static_cast<int>(gridDim.x) / CL;
  const int m_blocks = (M + Sh::TILE_M - 1) / Sh::TILE_M;
  const int n_blocks = (N + BN - 1) / BN;
  const int tiles = m_blocks * n_blocks;
  const int kt = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar->full[s], 1);
      mbar_init(&bar->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bar->acc_full[a], 1);
      mbar_init(&bar->acc_empty[a], Sh::CTAS * Sh::EPI_WARPS);
    }
    mbar_init(&bar->drain, 1);
    mbar_init(&bar->xfull, Sh::EPI_THREADS);    // every epilogue thread of the sending CTA
    mbar_init(&bar->xempty, Sh::EPI_THREADS);   // every epilogue thread of the receiving CTA
    bar->ctl.abort = 0;
    bar->consumed_hi = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&bar->tmem_base, Sh::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bar->tmem_base, Sh::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR)
    cluster_sync();   // both CTAs' barriers initialised and TMEM allocated before any cross-CTA signal
  else
    __syncthreads();
  tc_fence_after();
  // Launched as a programmatic dependent, the set-up above overlaps the tail
  // of the previous kernel; from here on the operands, C and the stream-K
  // workspace may be touched only once that kernel has completed.
  pdl_launch_dependents();
  WorkIter it;
  it.init(sk, kt, worker, workers);
  int tile, k0, k1;
  // the work items of this CTA (KX: this pair's half of each tile's K-loop)
  auto next_item = [&](int& t_, int& a_, int& b_) {
    if (!it.next(t_, a_, b_)) return false;
    if (KX) {
      const int h = (kt + 1) / 2;
      if (pidx == 0) b_ = h; else a_ = h;
    }
    return true;
  };
  // While the previous kernel finishes, bring the first ring-full of this
  // CTA's operand boxes into L2: a prefetch writes nothing and the L2 stays
  // coherent with any write the previous kernel still makes, so it needs no
  // wait; the loads after the wait then start from L2.  (Measured, back-to-back
  // launches with a pause between samples: FP16 4096^3 81.70 -> 81.46 us,
  // BF16 8192^2 x 256 35.32 -> 34.71 us, BF16 8192 x 128 x 8192 31.78 ->
  // 31.51 us; bit-identical results.)
  if (!ctl.inputs_ready && warp == 0 && lane == 0) {
    WorkIter pf = it;
    int t_, a_, b_;
    int left = stages;
    auto pf_next = [&](int& tt, int& aa, int& bb) {
      if (!pf.next(tt, aa, bb)) return false;
      if (KX) {
        const int h = (kt + 1) / 2;
        if (pidx == 0) bb = h; else aa = h;
      }
      return true;
    };
    while (left > 0 && pf_next(t_, a_, b_)) {
      int mb, nb;
      tile_coords(t_, m_blocks, n_blocks, mb, nb, sk.raster_gm);
      const int m_row = mb * Sh::TILE_M + rank * Sh::A_ROWS;
      const int n_row = nb * BN + rank * Sh::B_ROWS;
      for (int kb = a_; kb < b_ && left > 0; ++kb, --left) {
        tma_prefetch_l2_2d(&tmA, kb * BK, m_row);
        tma_prefetch_l2_2d(&tmB, kb * BK, n_row);
      }
    }
  }
  // With the caller's promise that nothing in flight writes A or B, the
  // producer and the MMA issuer start while the previous kernel is still
  // finishing; only the epilogue (C, the stream-K workspace) waits for it.
  if (!ctl.inputs_ready) pdl_wait();
  const uint32_t tmem = bar->tmem_base;
  CtaCtl* cta = &bar->ctl;
  int issued = 0;  // producer only

  if (warp == 0) {
    // ---------------- producer (every CTA) ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      const uint64_t keep_a = l2_policy_keep();
      int held_nb = -1;   // N block whose B tile fills the ring's B halves, slot kb holding K step kb
      while (!cta->abort && next_item(tile, k0, k1)) {
        int mb, nb;
        tile_coords(tile, m_blocks, n_blocks, mb, nb, sk.raster_gm);
        const int m_row = mb * Sh::TILE_M + rank * Sh::A_ROWS;
        const int n_row = nb * BN + rank * Sh::B_ROWS;
        // A whole K-loop in a ring of exactly kt slots puts K step kb in slot kb
        // for every tile, so a repeated N block finds its B tile still there: no
        // write ever reaches a slot's B half while that is so.
        const bool whole_ring = !PAIR && sk.b_resident && k0 == 0 && k1 == kt && kt == stages && s == 0;
        const bool keep_b = whole_ring && nb == held_nb;
        held_nb = whole_ring ? nb : -1;
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(&bar->empty[s], ph ^ 1u, ctl, cta, kSiteProducerEmpty)) goto producer_done;
          uint8_t* slot = ring + s * STAGE;
          if (PAIR) {
            if (leader) mbar_arrive_expect_tx(&bar->full[s], 2 * STAGE);
            const uint32_t full_leader = mapa_shared(smem_u32(&bar->full[s]), lead_rank);
            tma_load_2d_pair_keep(smem_u32(slot), &tmA, full_leader, kb * BK, m_row, keep_a);
            tma_load_2d_pair(smem_u32(slot + Sh::A_BYTES), &tmB, full_leader, kb * BK, n_row);
            ++issued;
          } else if (!(ctl.inject_lost_load && tile == tiles - 1 && kb == kt - 1)) {
            mbar_arrive_expect_tx(&bar->full[s], keep_b ? Sh::A_BYTES : STAGE);
            tma_load_2d_keep(smem_u32(slot), &tmA, &bar->full[s], kb * BK, m_row, keep_a);
            if (!keep_b) tma_load_2d(smem_u32(slot + Sh::A_BYTES), &tmB, &bar->full[s], kb * BK, n_row);
            ++issued;
          }
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread; the even CTA of a pair) ----------------
    if (lane == 0 && leader) {
      int s = 0;
      uint32_t ph = 0;
      int consumed = 0;
      for (int t = 0; next_item(tile, k0, k1); ++t) {
        const int a = t & 1;
        if (!mbar_wait(&bar->acc_empty[a], ((t >> 1) & 1) ^ 1u, ctl, cta, kSiteMmaAccEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem + a * BN;
        bool ok = true;
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(&bar->full[s], ph, ctl, cta, kSiteConsumerFull)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(ring + s * STAGE);
          const uint64_t da = umma_desc_sw128(a_addr);
          const uint64_t db = umma_desc_sw128(a_addr + Sh::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // advancing the start address by 32 bytes (>> 4 = 2) steps 16 elements along K
            const uint32_t acc = (kb == k0 && kk == 0) ? 0u : 1u;
            if (PAIR)
              umma_f16_pair(d, da + 2 * kk, db + 2 * kk, IDESC, acc);
            else
              umma_f16(d, da + 2 * kk, db + 2 * kk, IDESC, acc);
          }
          // slot s is free (in every CTA that loaded into it) once these MMAs have read it
          if (PAIR) umma_commit_pair(&bar->empty[s], pair_mask); else umma_commit(&bar->empty[s]);
          ++consumed;
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        if (PAIR) umma_commit_pair(&bar->acc_full[a], pair_mask); else umma_commit(&bar->acc_full[a]);
      }
      bar->consumed_hi = consumed;
      // every MMA issued by this thread has completed once drain fires
      if (PAIR) umma_commit_pair(&bar->drain, static_cast<uint16_t>(1u << lead_rank)); else umma_commit(&bar->drain);
      CtaCtl never_abort{0};
      mbar_wait(&bar->drain, 0, ctl, &never_abort, kSiteDrain);
    }
  } else {
    // ---------------- epilogue (warps 2..5 of every CTA) ----------------
    if (ctl.inputs_ready) pdl_wait();
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int e = warp - 2;
    const int row = q * 32 + lane;      // accumulator row of this CTA that this thread holds
    const int c_begin = (e >> 2) * Sh::WARP_CHUNKS;   // this warp's 64-column chunks
    const int c_end = c_begin + Sh::WARP_CHUNKS;
    uint8_t* my_stage = epi + e * Sh::EPI_BUFS * kUmmaEpiBufBytes;
    int sb = 0;
    for (int t = 0; next_item(tile, k0, k1); ++t) {
      int mb, nb;
      tile_coords(tile, m_blocks, n_blocks, mb, nb, sk.raster_gm);
      const int a = t & 1;
      // A split tile (stream-K): every segment stores its FP32 partial; the
      // segment that completes last sums all of them in K order and writes C.
      const bool split = !KX && ((k0 > 0) || (k1 < kt));
      SplitTile sp;
      if (split) sp.init(tile, kt, sk, workers, CL, crank);
      uint32_t ok = 1;
      if (lane == 0) ok = mbar_wait(&bar->acc_full[a], (t >> 1) & 1, ctl, cta, kSiteEpilogueAccFull) ? 1u : 0u;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // one decision for all four epilogue warps (they meet at named barriers below)
      // Fast path of a split tile: the owner of its first K step (normally the
      // segment that completes last) sees every other segment counted within
      // kSkPollNs, adds their partials to its own accumulator and writes C
      // directly.  Otherwise it falls back to the counted path below, which
      // never waits, so no CTA depends on another being resident.
      if (split && e == 0 && lane == 0) {
        bar->sk_last = (worker == sp.w_first && sp.poll_others(sk.epoch)) ? 2 : 0;
        __threadfence();
      }
      if (!epi_bar_and<Sh::EPI_THREADS>(ok != 0 && !cta->abort)) break;
      const bool fast = split && bar->sk_last == 2;
      tc_fence_after();
      const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * BN;
      const int y = mb * Sh::TILE_M + rank * Sh::A_ROWS + q * 32;
      const int x0 = nb * BN;   // first column of this pair's tile
      if (KX) {
        // K split over the two pairs: pair 1 sends its FP32 half of the
        // accumulator to the CTA of the same pair rank in pair 0 (row-
        // innermost float4 groups, conflict-free), which adds it to its own
        // half and writes C.  xfull / xempty hand the 64 KB buffer back and forth.
        const uint32_t xph = static_cast<uint32_t>(t & 1);
        const bool xok = pidx == 1 ? mbar_wait_acq_cluster(&bar->xempty, xph ^ 1u, ctl, cta, kSiteKSplitXfer)
                                   : mbar_wait_acq_cluster(&bar->xfull, xph, ctl, cta, kSiteKSplitXfer);
        if (!epi_bar_and<Sh::EPI_THREADS>(xok && !cta->abort)) break;
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
          uint32_t v[64];
          load_acc_chunk(trow + c * kUmmaEpiCols, v);
          if (c == c_end - 1) {
            // all of accumulator a is in registers: hand it back to the MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&bar->acc_empty[a]), lead_rank));
          }
          float4* xb = xbuf + static_cast<size_t>(c) * 16 * Sh::A_ROWS + row;
          if (pidx == 1) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              st_cluster_f4(mapa_shared(smem_u32(xb + i * Sh::A_ROWS), crank - 2u),
                            make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                        __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
            continue;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 p = xb[i * Sh::A_ROWS];
            v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) + p.x);
            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + p.y);
            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + p.z);
            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + p.w);
          }
          if (lane == 0) bulk_wait_read<Sh::EPI_BUFS - 1>();
          __syncwarp();
          const int x = x0 + c * kUmmaEpiCols;
          stage_and_store<BF16>(v, my_stage + sb * kUmmaEpiBufBytes, lane, &tmC, x, y, (x < N) && (y < M));
          if (++sb == Sh::EPI_BUFS) sb = 0;
        }
        // release: the sent half is visible to pair 0 / the buffer may be refilled
        if (pidx == 1)
          mbar_arrive_cluster(mapa_shared(smem_u32(&bar->xfull), crank - 2u));
        else
          mbar_arrive_cluster(mapa_shared(smem_u32(&bar->xempty), crank + 2u));
        continue;
      }
      if (!split) {
        // Whole tile: the TMEM load of chunk c + 1 is in flight while chunk c
        // is converted, staged and stored (chunks unrolled, so no register
        // that a load is still filling is carried around a loop).
        uint32_t v[64];
        issue_acc_chunk(trow + c_begin * kUmmaEpiCols, v);
#pragma unroll
        for (int j = 0; j < Sh::WARP_CHUNKS; ++j) {
          const int c = c_begin + j;
          tmem_wait_ld();
          regs_after_wait(v);
          uint32_t pk[32];
          pack_chunk<BF16>(v, pk);
          if (j + 1 < Sh::WARP_CHUNKS) {
            issue_acc_chunk(trow + (c + 1) * kUmmaEpiCols, v);
          } else {
            // all of accumulator a has been read: hand it back to the MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (PAIR)
                mbar_arrive_cluster(mapa_shared(smem_u32(&bar->acc_empty[a]), lead_rank));
              else
                mbar_arrive(&bar->acc_empty[a]);
            }
          }
          if (lane == 0) bulk_wait_read<Sh::EPI_BUFS - 1>();
          __syncwarp();
          const int x = x0 + c * kUmmaEpiCols;
          store_packed(pk, my_stage + sb * kUmmaEpiBufBytes, lane, &tmC, x, y, (x < N) && (y < M));
          if (++sb == Sh::EPI_BUFS) sb = 0;
        }
        continue;
      }
#pragma unroll 1
      for (int c = c_begin; c < c_end; ++c) {
        uint32_t v[64];
        load_acc_chunk(trow + c * kUmmaEpiCols, v);
        if (c == c_end - 1) {
          // all of accumulator a is in registers: hand it back to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (PAIR)
              mbar_arrive_cluster(mapa_shared(smem_u32(&bar->acc_empty[a]), lead_rank));
            else
              mbar_arrive(&bar->acc_empty[a]);
          }
        }
        if (fast) {
          // own segment first (it holds K step 0), then the others in K order
          for (int w = sp.w_first + 1; w <= sp.w_last; ++w) {
            if (!sp.has_segment(w)) continue;
            const float4* src = reinterpret_cast<const float4*>(sk.workspace) +
                                partial_at<BN>(sp.slot(w, CL, crank), c, 0, row);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float4 p = __ldcg(src + i * Sh::A_ROWS);
              v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) + p.x);
              v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + p.y);
              v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + p.z);
              v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + p.w);
            }
          }
        } else if (split) {
          float4* dst = reinterpret_cast<float4*>(sk.workspace) + partial_at<BN>(sp.slot(worker, CL, crank), c, 0, row);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            __stcg(dst + i * Sh::A_ROWS, make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
          continue;
        }
        if (lane == 0) bulk_wait_read<Sh::EPI_BUFS - 1>();
        __syncwarp();
        const int x = x0 + c * kUmmaEpiCols;
        stage_and_store<BF16>(v, my_stage + sb * kUmmaEpiBufBytes, lane, &tmC, x, y, (x < N) && (y < M));
        if (++sb == Sh::EPI_BUFS) sb = 0;
      }
      if (!split || fast) continue;
      // count this segment in; the tile's counter is tagged with the launch epoch
      __threadfence();
      epi_bar_sync<Sh::EPI_THREADS>();
      if (e == 0 && lane == 0) {
        bar->sk_last = sp.count_in(sk.epoch) ? 1 : 0;
        __threadfence();
      }
      epi_bar_sync<Sh::EPI_THREADS>();
      if (!bar->sk_last) continue;
#pragma unroll 1
      for (int c = c_begin; c < c_end; ++c) {
        uint32_t v[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = 0u;
        bool first = true;
        for (int w = sp.w_first; w <= sp.w_last; ++w) {
          if (!sp.has_segment(w)) continue;
          const float4* src = reinterpret_cast<const float4*>(sk.workspace) +
                              partial_at<BN>(sp.slot(w, CL, crank), c, 0, row);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 p = __ldcg(src + i * Sh::A_ROWS);
            if (first) {
              v[4 * i] = __float_as_uint(p.x);
              v[4 * i + 1] = __float_as_uint(p.y);
              v[4 * i + 2] = __float_as_uint(p.z);
              v[4 * i + 3] = __float_as_uint(p.w);
            } else {
              v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) + p.x);
              v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + p.y);
              v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + p.z);
              v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + p.w);
            }
          }
          first = false;
        }
        if (lane == 0) bulk_wait_read<Sh::EPI_BUFS - 1>();
        __syncwarp();
        const int x = x0 + c * kUmmaEpiCols;
        stage_and_store<BF16>(v, my_stage + sb * kUmmaEpiBufBytes, lane, &tmC, x, y, (x < N) && (y < M));
        if (++sb == Sh::EPI_BUFS) sb = 0;
      }
    }
    if (lane == 0) bulk_wait<0>();
  }

  __syncthreads();
  if (cta->abort && warp == 0 && lane == 0) {
    CtaCtl never_abort{0};
    if (PAIR) {
      // this CTA's loads count on the even CTA's barrier: give any still in
      // flight time to land before the pair tears down
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 200000ull) __nanosleep(1000);
    } else {
      // loads still in flight land in shared memory: wait for them before exit
      for (int i = bar->consumed_hi; i < issued; ++i)
        mbar_wait(&bar->full[i % stages], static_cast<uint32_t>((i / stages) & 1), ctl, &never_abort, kSiteDrain);
    }
  }
  if (PAIR) {
    tc_fence_before();
    cluster_sync();   // the even CTA's MMAs, which touch both CTAs, have completed
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem, Sh::TMEM_COLS); else tmem_dealloc(tmem, Sh::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// exact INT8 x INT8 -> INT32 on the tcgen05 tensor cores
// ---------------------------------------------------------------------------
// sm_103a has no integer kind of tcgen05.mma.  Every int8 value is exact in
// FP16 and every product of two of them (|p| <= 2^14) is exact in FP32, so the
// FP16 kind computes integer products exactly; an FP32 sum of such products
// stays exact while its magnitude stays within 2^24, i.e. over at most
// 2^24 / 2^14 = 1024 products.  The MMA therefore restarts the accumulator
// every kI8ChunkSteps K steps (1024 elements), alternating the two TMEM
// buffers, and the epilogue warps convert each finished chunk to int32 and add
// it to a running int32 sum held in registers (wrapping modulo 2^32, as the
// definition does).  The operands are converted to FP16 in global memory first
// (i8_to_f16_kernel): converting inside the ring would triple the
// shared-memory traffic per MMA.  Tile: 256 x 256 per CTA pair (each CTA
// 128 rows of A and 128 of B, as for FP16); a last wave at most half full
// runs as 256 x 128 half tiles (I8Item), and K-loops are split (stream-K,
// exact int32 partials) only when the tiles do not fill one wave.
constexpr int kI8ChunkSteps = 1024 / BK;   // 16 K steps of 64

// Four int8 values (one 32-bit word) to four FP16 values, exactly.  With the
// sign bit flipped, byte b holds u = x + 128 in [0, 255]; the FP16 bit pattern
// 0x64 : u is 1024 + u (FP16 spacing is 1 on [1024, 2048)), so one byte
// permute builds two such halves and subtracting 1152 = 1024 + 128 returns x
// with no rounding.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t p01 = __byte_perm(u, 0x64646464u, 0x5140);   // bytes u0, 0x64, u1, 0x64
  const uint32_t p23 = __byte_perm(u, 0x64646464u, 0x5342);   // bytes u2, 0x64, u3, 0x64
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
  __half2 h01 = __hsub2(*reinterpret_cast<const __half2*>(&p01), bias);
  __half2 h23 = __hsub2(*reinterpret_cast<const __half2*>(&p23), bias);
  lo = *reinterpret_cast<uint32_t*>(&h01);
  hi = *reinterpret_cast<uint32_t*>(&h23);
}

// The FP16 copies (64 MiB at 4096^3, half the L2) are read by the GEMM right
// after: they are stored with an L2 evict-last hint, so that more of them are
// still in L2 when it starts and their write-back can wait for its MMAs.
// (Measured per INT8 call, interleaved, bit-identical: 4096^3 109.8 -> 108.9
// us, 4096 x 6144 x 4096 154.6 -> 154.1 us, 8192^2 x 4096 334.1 -> 333.3 us.
// The same hint on the GEMM's loads of A added nothing.)
__device__ __forceinline__ void i8x16_store_f16(const uint4 raw, uint4* dst) {
  uint32_t h[8];
  i8x4_to_f16x4(raw.x, h[0], h[1]);
  i8x4_to_f16x4(raw.y, h[2], h[3]);
  i8x4_to_f16x4(raw.z, h[4], h[5]);
  i8x4_to_f16x4(raw.w, h[6], h[7]);
  const uint64_t keep = l2_policy_keep();
  st_global_v4_hint(dst, h[0], h[1], h[2], h[3], keep);
  st_global_v4_hint(dst + 1, h[4], h[5], h[6], h[7], keep);
}

// A then B, 16 int8 values per step of a grid-stride loop that keeps two
// 16-byte loads in flight per thread; the FP16 copies are written with
// L2-allocating, evict-last stores, since the GEMM reads them next.
__global__ void __launch_bounds__(256) i8_to_f16_kernel(const int8_t* __restrict__ a, __half* __restrict__ a16,
                                                        int64_t na16, const int8_t* __restrict__ b,
                                                        __half* __restrict__ b16, int64_t nb16) {
  const int64_t total = na16 + nb16;   // 16-element groups
  pdl_launch_dependents();   // the GEMM may start its set-up; it waits for this grid before reading
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  auto src = [&](int64_t i) {
    return i < na16 ? reinterpret_cast<const uint4*>(a) + i : reinterpret_cast<const uint4*>(b) + (i - na16);
  };
  auto dst = [&](int64_t i) {
    return i < na16 ? reinterpret_cast<uint4*>(a16) + 2 * i : reinterpret_cast<uint4*>(b16) + 2 * (i - na16);
  };
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + stride < total; i += 2 * stride) {
    const uint4 r0 = __ldcs(src(i));
    const uint4 r1 = __ldcs(src(i + stride));
    i8x16_store_f16(r0, dst(i));
    i8x16_store_f16(r1, dst(i + stride));
  }
  if (i < total) i8x16_store_f16(__ldcs(src(i)), dst(i));
}

// The same conversion launched early: a programmatic dependent of the
// previous call's GEMM (when the caller promised that this call's inputs were
// final before that call), so that it runs beside that GEMM's CTAs.  Measured
// on GB300 beside the INT8 pair kernel (10 warps x 168 registers and all but
// 2 KB of shared memory per SM): one more block of at most two warps starts
// on each SM (a four-warp block does not), and a finished block is not
// replaced there until the GEMM ends.  So the grid is one persistent two-warp
// block per SM, with eight 16-byte loads in flight per thread.  Only the last
// block waits for the previous GEMM before it exits, so that this grid, and
// what waits for it, completes after that GEMM.
constexpr int kEarlyConvThreads = 64;
constexpr int kEarlyConvDepth = 8;
__global__ void __launch_bounds__(kEarlyConvThreads) i8_to_f16_early_kernel(
    const int8_t* __restrict__ a, __half* __restrict__ a16, int64_t na16, const int8_t* __restrict__ b,
    __half* __restrict__ b16, int64_t nb16) {
  const int64_t total = na16 + nb16;   // 16-element groups
  pdl_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  auto src = [&](int64_t i) {
    return i < na16 ? reinterpret_cast<const uint4*>(a) + i : reinterpret_cast<const uint4*>(b) + (i - na16);
  };
  auto dst = [&](int64_t i) {
    return i < na16 ? reinterpret_cast<uint4*>(a16) + 2 * i : reinterpret_cast<uint4*>(b16) + 2 * (i - na16);
  };
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += kEarlyConvDepth * stride) {
    uint4 r[kEarlyConvDepth];
#pragma unroll
    for (int d = 0; d < kEarlyConvDepth; ++d)
      if (i + d * stride < total) r[d] = __ldcs(src(i + d * stride));
#pragma unroll
    for (int d = 0; d < kEarlyConvDepth; ++d)
      if (i + d * stride < total) i8x16_store_f16(r[d], dst(i + d * stride));
  }
  if (blockIdx.x == gridDim.x - 1) pdl_wait();
}

// Store one 32-row x 32-column INT32 chunk through a 4 KB swizzled staging
// buffer and a TMA store (lane t holds row t).
__device__ __forceinline__ void stage_and_store_i32(const uint32_t* v, uint8_t* buf, int lane, const CUtensorMap* tmap_c,
                                                    int x, int y, bool in_bounds) {
  const uint32_t base = smem_u32(buf);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + sw128_offset(lane, j)), "r"(v[4 * j]),
                 "r"(v[4 * j + 1]), "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                 : "memory");
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && in_bounds) tma_store_2d(tmap_c, base, x, y);
  if (lane == 0) bulk_commit();
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Threads: warp 0 TMA producer, warp 1 MMA issuer, warps 2..9 epilogue.
// Epilogue warp w reads TMEM lane quarter w % 4 and column half (w - 2) / 4,
// so each thread keeps the int32 running sums of 128 accumulator columns.
constexpr int kI8EpiWarps = 8;
constexpr int kI8Threads = 64 + 32 * kI8EpiWarps;

__device__ __forceinline__ bool i8_epi_bar_and(bool pred) {   // the 8 epilogue warps only
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return r != 0;
}

// Work item of the INT8 pair kernel: items below half_from are whole 256 x 256
// tiles (tile = item); each tile from half_from on is split along N into two
// 256 x 128 items (the last partial wave of whole tiles would otherwise leave
// most pairs idle: half tiles spread it over twice as many pairs, with no
// partial sums to combine).
struct I8Item {
  int mb, n0;     // 256-row block; first column
  bool half;      // 128 columns instead of 256
  __device__ __forceinline__ void decode(int item, int half_from, int m_blocks, int n_blocks, int gm) {
    int tile = item, hs = 0;
    half = item >= half_from;
    if (half) {
      tile = half_from + (item - half_from) / 2;
      hs = (item - half_from) & 1;
    }
    int nb;
    tile_coords(tile, m_blocks, n_blocks, mb, nb, gm);
    n0 = nb * 256 + hs * 128;
  }
};

template <bool PAIR>
__global__ void __launch_bounds__(kI8Threads, 1)
    umma_i8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmBh, int M, int N,
                   int K, int stages, KernelCtl ctl, SkParams sk, int half_from) {
  constexpr int BN = 256;
  constexpr int HALF = BN / 2;   // columns per epilogue thread
  using Sh = RingShape<BN, PAIR>;
  constexpr int STAGE = Sh::STAGE;
  constexpr uint32_t IDESC = umma_idesc_f16(false, Sh::TILE_M, BN);
  constexpr uint32_t IDESC_HALF = umma_idesc_f16(false, Sh::TILE_M, BN / 2);
  static_assert(kI8EpiWarps * kUmmaEpiBufBytes <= kUmmaEpiBytes, "staging region too small");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* epi = smem + stages * STAGE;
  UmmaBarriers* bar = reinterpret_cast<UmmaBarriers*>(epi + kUmmaEpiBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int worker = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int workers = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int m_blocks = (M + Sh::TILE_M - 1) / Sh::TILE_M;
  const int n_blocks = (N + BN - 1) / BN;
  const int kt = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar->full[s], 1);
      mbar_init(&bar->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bar->acc_full[a], 1);
      mbar_init(&bar->acc_empty[a], Sh::CTAS * kI8EpiWarps);
    }
    mbar_init(&bar->drain, 1);
    bar->ctl.abort = 0;
    bar->consumed_hi = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&bar->tmem_base, Sh::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bar->tmem_base, Sh::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();
  pdl_wait();   // the FP16 copies are written by the conversion kernel launched just before
  // Only now may a dependent (an early conversion for the next call) start:
  // the copy buffer it writes is free once the GEMM before this one is done.
  pdl_launch_dependents();
  const uint32_t tmem = bar->tmem_base;
  CtaCtl* cta = &bar->ctl;
  int issued = 0;
  WorkIter it;
  it.init(sk, kt, worker, workers);
  int tile, k0, k1;

  if (warp == 0) {
    // ---------------- producer (every CTA) ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      while (!cta->abort && it.next(tile, k0, k1)) {
        I8Item w;
        w.decode(tile, half_from, m_blocks, n_blocks, sk.raster_gm);
        const int m_row = w.mb * Sh::TILE_M + rank * Sh::A_ROWS;
        // a half item: each CTA of the pair loads 64 of its 128 B rows
        const int n_row = w.n0 + rank * (w.half ? Sh::B_ROWS / 2 : Sh::B_ROWS);
        const uint32_t tx_bytes = w.half ? 2 * (Sh::A_ROWS + Sh::B_ROWS / 2) * BK * 2 : 2 * STAGE;
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(&bar->empty[s], ph ^ 1u, ctl, cta, kSiteProducerEmpty)) goto i8_producer_done;
          uint8_t* slot = ring + s * STAGE;
          if (PAIR) {
            if (leader) mbar_arrive_expect_tx(&bar->full[s], tx_bytes);
            const uint32_t full_leader = mapa_shared(smem_u32(&bar->full[s]), 0);
            tma_load_2d_pair(smem_u32(slot), &tmA, full_leader, kb * BK, m_row);
            tma_load_2d_pair(smem_u32(slot + Sh::A_BYTES), w.half ? &tmBh : &tmB, full_leader, kb * BK, n_row);
          } else {
            mbar_arrive_expect_tx(&bar->full[s], STAGE);
            tma_load_2d(smem_u32(slot), &tmA, &bar->full[s], kb * BK, m_row);
            tma_load_2d(smem_u32(slot + Sh::A_BYTES), &tmB, &bar->full[s], kb * BK, n_row);
          }
          ++issued;
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
    i8_producer_done:;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: one accumulator buffer per 1024-element chunk of K ----------------
    if (lane == 0 && leader) {
      int s = 0;
      uint32_t ph = 0;
      int consumed = 0;
      int t = 0;
      bool ok = true;
      while (ok && it.next(tile, k0, k1)) {
        const uint32_t idesc = (PAIR && tile >= half_from) ? IDESC_HALF : IDESC;   // N = 128 for a half item
        // chunks of at most kI8ChunkSteps K steps from k0: each FP32 sum stays exact
        for (int kb0 = k0; kb0 < k1 && ok; kb0 += kI8ChunkSteps, ++t) {
          const int a = t & 1;
          if (!mbar_wait(&bar->acc_empty[a], ((t >> 1) & 1) ^ 1u, ctl, cta, kSiteMmaAccEmpty)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + a * BN;
          const int kb1 = min(k1, kb0 + kI8ChunkSteps);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&bar->full[s], ph, ctl, cta, kSiteConsumerFull)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(ring + s * STAGE);
            const uint64_t da = umma_desc_sw128(a_addr);
            const uint64_t db = umma_desc_sw128(a_addr + Sh::A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              const uint32_t acc = (kb == kb0 && kk == 0) ? 0u : 1u;
              if (PAIR)
                umma_f16_pair(d, da + 2 * kk, db + 2 * kk, idesc, acc);
              else
                umma_f16(d, da + 2 * kk, db + 2 * kk, IDESC, acc);
            }
            if (PAIR) umma_commit_pair(&bar->empty[s], 0x3); else umma_commit(&bar->empty[s]);
            ++consumed;
            if (++s == stages) { s = 0; ph ^= 1u; }
          }
          if (!ok) break;
          if (PAIR) umma_commit_pair(&bar->acc_full[a], 0x3); else umma_commit(&bar->acc_full[a]);
        }
      }
      bar->consumed_hi = consumed;
      if (PAIR) umma_commit_pair(&bar->drain, 0x1); else umma_commit(&bar->drain);
      CtaCtl never_abort{0};
      mbar_wait(&bar->drain, 0, ctl, &never_abort, kSiteDrain);
    }
  } else {
    // ---------------- epilogue: int32 running sum of the exact FP32 chunk sums ----------------
    const int q = warp & 3;
    const int e = warp - 2;
    const int h = e >> 2;              // column half of the accumulator
    const int row = q * 32 + lane;     // accumulator row of this CTA that this thread holds
    uint8_t* my_stage = epi + e * kUmmaEpiBufBytes;
    int t = 0;
    bool ok = true;
    while (ok && it.next(tile, k0, k1)) {
      I8Item wi;
      wi.decode(tile, half_from, m_blocks, n_blocks, sk.raster_gm);
      const int mb = wi.mb;
      const int cols = wi.half ? HALF / 2 : HALF;   // accumulator columns of this thread
      // A split tile (stream-K): each segment's int32 partial is exact, so the
      // order in which the segments are added does not change the result.
      const bool split = (k0 > 0) || (k1 < kt);
      uint32_t sum[HALF];
#pragma unroll
      for (int i = 0; i < HALF; ++i) sum[i] = 0u;
      for (int kb0 = k0; kb0 < k1; kb0 += kI8ChunkSteps, ++t) {
        const int a = t & 1;
        uint32_t w = 1;
        if (lane == 0) w = mbar_wait(&bar->acc_full[a], (t >> 1) & 1, ctl, cta, kSiteEpilogueAccFull) ? 1u : 0u;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!i8_epi_bar_and(w != 0 && !cta->abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * BN + h * cols;
#pragma unroll
        for (int sub = 0; sub < HALF / 16; ++sub) {   // 16 columns at a time: sum[] holds 128 registers
          if (sub * 16 >= cols) break;
          uint32_t v[16];
          tmem_ld_32x32b_x16(trow + sub * 16, v);
          tmem_wait_ld();
          regs_after_wait(v);
#pragma unroll
          for (int i = 0; i < 16; ++i)   // exact integers of magnitude <= 2^24 in FP32
            sum[sub * 16 + i] += static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR)
            mbar_arrive_cluster(mapa_shared(smem_u32(&bar->acc_empty[a]), 0));
          else
            mbar_arrive(&bar->acc_empty[a]);
        }
      }
      if (!ok) break;
      if (split) {
        SplitTile sp;
        sp.init(tile, kt, sk, workers, Sh::CTAS, rank);
        // first-K-step owner: take the fast path if every other segment is in
        if (e == 0 && lane == 0) {
          bar->sk_last = (worker == sp.w_first && sp.poll_others(sk.epoch)) ? 2 : 0;
          __threadfence();
        }
        i8_epi_bar_and(true);
        const bool fast = bar->sk_last == 2;
        if (!fast) {
          // store this segment's partial, count it in; the last one adds them all
          uint4* dst = reinterpret_cast<uint4*>(sk.workspace);
          const int my = sp.slot(worker, Sh::CTAS, rank);
#pragma unroll
          for (int i = 0; i < HALF / 4; ++i)
            __stcg(dst + partial_at<BN>(my, 2 * h + i / 16, i % 16, row),
                   make_uint4(sum[4 * i], sum[4 * i + 1], sum[4 * i + 2], sum[4 * i + 3]));
          __threadfence();
          i8_epi_bar_and(true);
          if (e == 0 && lane == 0) {
            bar->sk_last = sp.count_in(sk.epoch) ? 1 : 0;
            __threadfence();
          }
          i8_epi_bar_and(true);
          if (!bar->sk_last) continue;
#pragma unroll
          for (int i = 0; i < HALF; ++i) sum[i] = 0u;
        }
        // add the other segments' partials (every segment, when counted in: its own included)
        for (int w2 = sp.w_first; w2 <= sp.w_last; ++w2) {
          if (!sp.has_segment(w2) || (fast && w2 == worker)) continue;
          const uint4* src = reinterpret_cast<const uint4*>(sk.workspace);
          const int sl = sp.slot(w2, Sh::CTAS, rank);
#pragma unroll
          for (int i = 0; i < HALF / 4; ++i) {
            const uint4 p = __ldcg(src + partial_at<BN>(sl, 2 * h + i / 16, i % 16, row));
            sum[4 * i] += p.x;
            sum[4 * i + 1] += p.y;
            sum[4 * i + 2] += p.z;
            sum[4 * i + 3] += p.w;
            if (i % 8 == 7) asm volatile("" ::: "memory");   // at most 8 loads in flight: sum[] keeps its registers
          }
        }
      }
      const int y = mb * Sh::TILE_M + rank * Sh::A_ROWS + q * 32;
#pragma unroll
      for (int sub = 0; sub < HALF / 32; ++sub) {
        if (sub * 32 >= cols) break;
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        const int x = wi.n0 + h * cols + sub * 32;
        stage_and_store_i32(sum + sub * 32, my_stage, lane, &tmC, x, y, (x < N) && (y < M));
      }
    }
    if (lane == 0) bulk_wait<0>();
  }

  __syncthreads();
  if (cta->abort && warp == 0 && lane == 0) {
    CtaCtl never_abort{0};
    if (PAIR) {
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 200000ull) __nanosleep(1000);
    } else {
      for (int i = bar->consumed_hi; i < issued; ++i)
        mbar_wait(&bar->full[i % stages], static_cast<uint32_t>((i / stages) & 1), ctl, &never_abort, kSiteDrain);
    }
  }
  if (PAIR) {
    tc_fence_before();
    cluster_sync();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem, Sh::TMEM_COLS); else tmem_dealloc(tmem, Sh::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// exact INT8 on tcgen05 with the int8 -> FP16 conversion overlapped in-kernel
// ---------------------------------------------------------------------------
// The same CTA-pair tile, TMA ring over FP16 copies of A and B, MMA sequence
// and int32 epilogue as umma_i8_kernel, but the copies are written by this
// kernel while it runs instead of by a conversion pass before it.
//
// Conversion units: one K step (64 columns) of one 128-row panel of A or of B,
// numbered K step major (unit u: K step u / P, panel u % P, P = ceil(M/128) +
// ceil(N/128) panels, A's first).  In every CTA a loader thread claims units
// (one, then four at a time) from a launch-wide counter (so the first K steps of every
// panel are converted first, and every unit is converted by whichever CTAs
// are resident: nothing depends on all CTAs running at once) and loads each
// into an int8 staging slot of shared memory with TMA.  Four converter warps
// read a slot, convert (i8x4_to_f16x4) and store the FP16 values with plain
// global stores; a signalling thread then counts the unit on its K step's
// counter (after a GPU-scope fence, one per group of units it finds ready).
// The TMA producer issues the loads of K step kb only once that counter holds
// all P units (then an acquire fence and a generic -> async proxy fence);
// from the first time it sees every K step complete it stops checking.  The
// counters come in two sets used by alternate launches: each launch zeroes
// the other set for the next one (which reads it only after this launch has
// completed).
//
// 512 threads = four warpgroups: converters (warps 0-3); TMA producer (warp
// 4), MMA issuer and TMEM owner (warp 5), signaller (warp 6), loader (warp
// 7); eight epilogue warps (8-15: TMEM lane quarter warp % 4, column half
// (warp - 8) / 4).  Launched at 128 registers per thread; the second
// warpgroup gives back to 48 and the epilogue warpgroups take 168 (their 128
// running int32 sums): 4*32*128 + 4*32*48 + 8*32*168 = 65,536.
constexpr int kOvThreads = 512;
constexpr int kConvWarps = 4;
constexpr int kOvLaunchRegs = 65536 / kOvThreads;   // what __launch_bounds__(512, 1) allows
constexpr int kOvCtlRegs = 48;
constexpr int kOvEpiRegs = 168;
static_assert(4 * 32 * kOvLaunchRegs + 4 * 32 * kOvCtlRegs + 8 * 32 * kOvEpiRegs <= kOvThreads * kOvLaunchRegs,
              "register split");
constexpr int kConvUnitRows = 128;    // rows of one unit (one CTA's half of a pair tile)
constexpr int kConvBatch = 4;         // units per claim
constexpr int kConvRing = 8;          // converted units the signaller may lag behind
static_assert(kConvUnitRows * BK == kI8ConvUnitBytes, "unit = 128 rows x one K step of int8");

struct ConvBarriers {
  uint64_t stg_full[kI8MaxStg];    // a unit's int8 tile landed (loader arrive + TMA bytes), or the end mark
  uint64_t stg_empty[kI8MaxStg];   // the converter warps have read it (count kConvWarps)
  uint64_t done[kConvRing];        // the converter warps stored a unit's FP16 values (count kConvWarps)
  uint64_t free[kConvRing];        // the signaller counted it (count 1)
  int32_t stg_unit[kI8MaxStg];     // unit in each staging slot; -1: no more units
  int32_t done_unit[kConvRing];    // unit in each hand-off slot; -1: the converters have finished
};
static_assert(sizeof(ConvBarriers) <= kI8ConvBarrierBytes, "conversion barrier region too small");

// Shape of the unit space of one launch.
struct ConvUnits {
  int pa, p, kt;               // A panels, all panels, K steps
  int64_t units;               // kt * p
  __device__ __forceinline__ void init(int M, int N, int K) {
    pa = (M + kConvUnitRows - 1) / kConvUnitRows;
    p = pa + (N + kConvUnitRows - 1) / kConvUnitRows;
    kt = (K + BK - 1) / BK;
    units = static_cast<int64_t>(kt) * p;
  }
  // K step, operand and first row of unit u
  __device__ __forceinline__ void coords(int64_t u, int& kb, bool& is_a, int& row0) const {
    kb = static_cast<int>(u / p);
    const int pn = static_cast<int>(u % p);
    is_a = pn < pa;
    row0 = (is_a ? pn : pn - pa) * kConvUnitRows;
  }
};

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__global__ void __launch_bounds__(kOvThreads, 1)
    umma_i8_overlap_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmA8,
                           const __grid_constant__ CUtensorMap tmB8, __half* a16, __half* b16, uint32_t* ctrs,
                           int kcap, uint32_t parity, int M, int N, int K, int stages, int stg_slots,
                           KernelCtl ctl) {
  constexpr int BN = 256;
  constexpr int HALF = BN / 2;
  using Sh = RingShape<BN, true>;
  constexpr int STAGE = Sh::STAGE;
  constexpr uint32_t IDESC = umma_idesc_f16(false, Sh::TILE_M, BN);
  static_assert(kI8EpiWarps * kUmmaEpiBufBytes <= kUmmaEpiBytes, "staging region too small");
  static_assert(Sh::A_ROWS == kConvUnitRows && Sh::B_ROWS == kConvUnitRows, "a unit is one CTA's half tile");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* stg = smem + stages * STAGE;
  uint8_t* epi = stg + stg_slots * kI8ConvUnitBytes;
  UmmaBarriers* bar = reinterpret_cast<UmmaBarriers*>(epi + kUmmaEpiBytes);
  ConvBarriers* cbar = reinterpret_cast<ConvBarriers*>(epi + kUmmaEpiBytes + kBarrierRegion);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int worker = static_cast<int>(blockIdx.x >> 1);
  const int workers = static_cast<int>(gridDim.x >> 1);
  const int m_blocks = (M + Sh::TILE_M - 1) / Sh::TILE_M;
  const int n_blocks = (N + BN - 1) / BN;
  const int tiles = m_blocks * n_blocks;
  ConvUnits cu;
  cu.init(M, N, K);
  const int kt = cu.kt;
  // counter set `parity`: a batch counter and kcap >= kt K-step counters, zero at launch
  uint32_t* claim_ctr = ctrs + parity * (kcap + 1);
  uint32_t* kstep_ctr = claim_ctr + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar->full[s], 1);
      mbar_init(&bar->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bar->acc_full[a], 1);
      mbar_init(&bar->acc_empty[a], 2 * kI8EpiWarps);
    }
    for (int g = 0; g < stg_slots; ++g) {
      mbar_init(&cbar->stg_full[g], 1);
      mbar_init(&cbar->stg_empty[g], kConvWarps);
    }
    for (int r = 0; r < kConvRing; ++r) {
      mbar_init(&cbar->done[r], kConvWarps);
      mbar_init(&cbar->free[r], 1);
    }
    mbar_init(&bar->drain, 1);
    bar->ctl.abort = 0;
    bar->consumed_hi = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc_pair(&bar->tmem_base, Sh::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 7 && lane == 0) {
    tma_prefetch_desc(&tmA8);
    tma_prefetch_desc(&tmB8);
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  pdl_launch_dependents();
  pdl_wait();   // A and B may come from the previous kernel; it may still read the FP16 copies
  const uint32_t tmem = bar->tmem_base;
  CtaCtl* cta = &bar->ctl;

  if (warp < kConvWarps) {
    // ---------------- converters (every CTA): staging slot -> FP16 copy -> signaller ----------------
    const int t = threadIdx.x;
    const int c = t & 3;
    const uint32_t stg0 = smem_u32(stg);
    int g = 0, r = 0;
    uint32_t gph = 0, fph = 0;
    for (;;) {
      // every lane observes the TMA bytes (acquire); the warp agrees on the outcome
      const bool w = mbar_wait(&cbar->stg_full[g], gph, ctl, cta, kSiteConvRing);
      if (!__all_sync(0xffffffffu, w)) break;
      const int32_t u = cbar->stg_unit[g];
      if (u >= 0) {
        const uint32_t sa = stg0 + static_cast<uint32_t>(g) * kI8ConvUnitBytes;
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ld_shared_v4(sa + static_cast<uint32_t>(((t >> 2) + 32 * i) * BK + c * 16));
        __syncwarp();
        if (lane == 0) mbar_arrive(&cbar->stg_empty[g]);
        int kb, row0;
        bool is_a;
        cu.coords(u, kb, is_a, row0);
        const int rows = is_a ? M : N;
        __half* dst = is_a ? a16 : b16;
        const int kx = kb * BK + c * 16;   // K % 16 == 0: a chunk is wholly inside or outside
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = row0 + (t >> 2) + 32 * i;
          if (row < rows && kx < K)
            i8x16_store_f16(v[i], reinterpret_cast<uint4*>(dst + static_cast<size_t>(row) * K + kx));
        }
      }
      if (++g == stg_slots) { g = 0; gph ^= 1u; }
      // hand the unit (or the end) to the signaller
      uint32_t ok = 1;
      if (lane == 0) ok = mbar_wait(&cbar->free[r], fph ^ 1u, ctl, cta, kSiteConvRing) ? 1u : 0u;
      if (__shfl_sync(0xffffffffu, ok, 0) == 0) break;
      __syncwarp();   // every lane's stores precede lane 0's release-arrive
      if (lane == 0) {
        if (warp == 0) cbar->done_unit[r] = u;
        mbar_arrive(&cbar->done[r]);
      }
      if (++r == kConvRing) { r = 0; fph ^= 1u; }
      if (u < 0) break;
    }
  } else if (warp < 8) {
    regs_decrease<kOvCtlRegs>();
    if (warp == 7 && lane == 0) {
      // ---------------- loader: claim units, TMA their int8 tiles into the staging ring ----------------
      if (blockIdx.x == 0) {   // the other counter set, for the next launch
        uint32_t* next_set = ctrs + (parity ^ 1u) * (kcap + 1);
        for (int i = 0; i <= kcap; ++i) next_set[i] = 0u;
      }
      int g = 0;
      uint32_t gph = 0;
      bool ok = true;
      // The counter counts units.  A CTA's first claim is one unit, so the first
      // K steps are spread over many CTAs and ready early; later claims take
      // kConvBatch units (fewer atomics).
      uint32_t b = atomicAdd(claim_ctr, 1u);
      uint32_t bn = 1;
      while (ok && b < cu.units) {
        const uint32_t b_next = atomicAdd(claim_ctr, static_cast<uint32_t>(kConvBatch));   // in flight meanwhile
        for (int i = 0; i < static_cast<int>(bn); ++i) {
          const int64_t u = static_cast<int64_t>(b) + i;
          if (u >= cu.units) break;
          if (!mbar_wait(&cbar->stg_empty[g], gph ^ 1u, ctl, cta, kSiteConvRing)) { ok = false; break; }
          int kb, row0;
          bool is_a;
          cu.coords(u, kb, is_a, row0);
          cbar->stg_unit[g] = static_cast<int32_t>(u);
          mbar_arrive_expect_tx(&cbar->stg_full[g], kI8ConvUnitBytes);
          tma_load_2d(smem_u32(stg + g * kI8ConvUnitBytes), is_a ? &tmA8 : &tmB8, &cbar->stg_full[g], kb * BK, row0);
          if (++g == stg_slots) { g = 0; gph ^= 1u; }
        }
        b = b_next;
        bn = kConvBatch;
      }
      if (ok && mbar_wait(&cbar->stg_empty[g], gph ^ 1u, ctl, cta, kSiteConvRing)) {
        cbar->stg_unit[g] = -1;   // end mark: a plain arrive completes the phase
        mbar_arrive(&cbar->stg_full[g]);
      }
    } else if (warp == 6 && lane == 0) {
      // ---------------- signaller: count converted units on their K steps ----------------
      int r = 0;
      uint32_t dph = 0;
      bool end = false;
      while (!end) {
        if (!mbar_wait(&cbar->done[r], dph, ctl, cta, kSiteConvRing)) break;
        // this unit and every later one already handed over, up to the end mark
        int n = 0;
        int rr = r;
        uint32_t pp = dph;
        for (;;) {
          if (cbar->done_unit[rr] < 0) { end = true; break; }
          ++n;
          if (++rr == kConvRing) { rr = 0; pp ^= 1u; }
          if (n == kConvRing || !mbar_try_wait(smem_u32(&cbar->done[rr]), pp)) break;
        }
        if (n == 0) break;
        __threadfence();   // release at GPU scope: the converters' stores, seen through the barriers
        for (int i = 0; i < n; ++i) {
          atomicAdd(kstep_ctr + cbar->done_unit[r] / cu.p, 1u);
          mbar_arrive(&cbar->free[r]);
          if (++r == kConvRing) { r = 0; dph ^= 1u; }
        }
      }
    } else if (warp == 4 && lane == 0) {
      // ---------------- producer (every CTA): a K step's loads once all its units are converted ----------------
      int s = 0;
      uint32_t ph = 0;
      int ready = 0;   // K steps [0, ready) are converted
      for (int tile = worker; tile < tiles; tile += workers) {
        int mb, nb;
        tile_coords(tile, m_blocks, n_blocks, mb, nb);
        const int m_row = mb * Sh::TILE_M + rank * Sh::A_ROWS;
        const int n_row = nb * BN + rank * Sh::B_ROWS;
        for (int kb = 0; kb < kt; ++kb) {
          if (kb >= ready) {
            const uint64_t t0 = global_timer_ns();
            for (;;) {
              uint32_t c[8];   // eight independent loads in flight
#pragma unroll
              for (int i = 0; i < 8; ++i)
                c[i] = ready + i < kt ? ld_volatile_u32(kstep_ctr + ready + i) : 0u;
              int adv = 0;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (adv == i && c[i] == static_cast<uint32_t>(cu.p)) adv = i + 1;
              ready += adv;
              if (kb < ready) break;
              if (cta->abort) goto ov_producer_done;
              if (global_timer_ns() - t0 > ctl.timeout_ns) {
                report_error(ctl, kDevErrTimeout, kSiteConvReady);
                cta->abort = 1;
                goto ov_producer_done;
              }
              __nanosleep(128);
            }
            __threadfence();             // acquire: the copies the counts stand for
            fence_proxy_async_global();  // written by generic stores, read by TMA
          }
          if (!mbar_wait(&bar->empty[s], ph ^ 1u, ctl, cta, kSiteProducerEmpty)) goto ov_producer_done;
          uint8_t* slot = ring + s * STAGE;
          if (leader) mbar_arrive_expect_tx(&bar->full[s], 2 * STAGE);
          const uint32_t full_leader = mapa_shared(smem_u32(&bar->full[s]), 0);
          tma_load_2d_pair(smem_u32(slot), &tmA, full_leader, kb * BK, m_row);
          tma_load_2d_pair(smem_u32(slot + Sh::A_BYTES), &tmB, full_leader, kb * BK, n_row);
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
    ov_producer_done:;
    } else if (warp == 5 && lane == 0 && leader) {
      // ---------------- MMA issuer: one accumulator buffer per 1024-element chunk of K ----------------
      int s = 0;
      uint32_t ph = 0;
      int t = 0;
      bool ok = true;
      for (int tile = worker; tile < tiles && ok; tile += workers) {
        for (int kb0 = 0; kb0 < kt && ok; kb0 += kI8ChunkSteps, ++t) {
          const int a = t & 1;
          if (!mbar_wait(&bar->acc_empty[a], ((t >> 1) & 1) ^ 1u, ctl, cta, kSiteMmaAccEmpty)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + a * BN;
          const int kb1 = min(kt, kb0 + kI8ChunkSteps);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&bar->full[s], ph, ctl, cta, kSiteConsumerFull)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(ring + s * STAGE);
            const uint64_t da = umma_desc_sw128(a_addr);
            const uint64_t db = umma_desc_sw128(a_addr + Sh::A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              umma_f16_pair(d, da + 2 * kk, db + 2 * kk, IDESC, (kb == kb0 && kk == 0) ? 0u : 1u);
            umma_commit_pair(&bar->empty[s], 0x3);
            if (++s == stages) { s = 0; ph ^= 1u; }
          }
          if (!ok) break;
          umma_commit_pair(&bar->acc_full[a], 0x3);
        }
      }
      umma_commit_pair(&bar->drain, 0x1);
      CtaCtl never_abort{0};
      mbar_wait(&bar->drain, 0, ctl, &never_abort, kSiteDrain);
    }
  } else {
    regs_increase<kOvEpiRegs>();
    // ---------------- epilogue: int32 running sum of the exact FP32 chunk sums ----------------
    const int q = warp & 3;
    const int e = warp - 8;
    const int h = e >> 2;              // column half of the accumulator
    uint8_t* my_stage = epi + e * kUmmaEpiBufBytes;
    int t = 0;
    bool ok = true;
    for (int tile = worker; tile < tiles && ok; tile += workers) {
      int mb, nb;
      tile_coords(tile, m_blocks, n_blocks, mb, nb);
      uint32_t sum[HALF];
#pragma unroll
      for (int i = 0; i < HALF; ++i) sum[i] = 0u;
      for (int kb0 = 0; kb0 < kt; kb0 += kI8ChunkSteps, ++t) {
        const int a = t & 1;
        uint32_t w = 1;
        if (lane == 0) w = mbar_wait(&bar->acc_full[a], (t >> 1) & 1, ctl, cta, kSiteEpilogueAccFull) ? 1u : 0u;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!i8_epi_bar_and(w != 0 && !cta->abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * BN + h * HALF;
#pragma unroll
        for (int sub = 0; sub < HALF / 16; ++sub) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(trow + sub * 16, v);
          tmem_wait_ld();
          regs_after_wait(v);
#pragma unroll
          for (int i = 0; i < 16; ++i)   // exact integers of magnitude <= 2^24 in FP32
            sum[sub * 16 + i] += static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&bar->acc_empty[a]), 0));
      }
      if (!ok) break;
      const int y = mb * Sh::TILE_M + rank * Sh::A_ROWS + q * 32;
#pragma unroll
      for (int sub = 0; sub < HALF / 32; ++sub) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        const int x = nb * BN + h * HALF + sub * 32;
        stage_and_store_i32(sum + sub * 32, my_stage, lane, &tmC, x, y, (x < N) && (y < M));
      }
    }
    if (lane == 0) bulk_wait<0>();
  }

  __syncthreads();
  // After an abort, give TMA loads still in flight and the partner's arrivals
  // on this CTA's barriers time to land before the pair tears down.
  if (cta->abort && threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) __nanosleep(1000);
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, Sh::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// register-staged ping-pong and no-overlap variants (256 threads, one tile per CTA)
// ---------------------------------------------------------------------------
constexpr int kPPThreads = 256;

// Global -> registers for one K step: A tile (128 rows) and B tile (BN rows),
// 16-byte chunks, zero outside the matrix.
template <int BN>
struct RegStage {
  static constexpr int A_CHUNKS = BM * 8 / kPPThreads;   // 4
  static constexpr int B_CHUNKS = BN * 8 / kPPThreads;   // BN/32
  uint4 a[A_CHUNKS];
  uint4 b[B_CHUNKS];

  __device__ __forceinline__ void load(const uint8_t* A, const uint8_t* B, int M, int N, int K, int m0, int n0, int kb) {
    const int tid = threadIdx.x;
    const int k0 = kb * BK;
#pragma unroll
    for (int i = 0; i < A_CHUNKS; ++i) {
      const int c = tid + i * kPPThreads;
      const int row = c >> 3, j = c & 7;
      const int gm = m0 + row, gk = k0 + j * 8;
      a[i] = make_uint4(0, 0, 0, 0);
      if (gm < M && gk < K) a[i] = __ldg(reinterpret_cast<const uint4*>(A + (static_cast<size_t>(gm) * K + gk) * 2));
    }
#pragma unroll
    for (int i = 0; i < B_CHUNKS; ++i) {
      const int c = tid + i * kPPThreads;
      const int row = c >> 3, j = c & 7;
      const int gn = n0 + row, gk = k0 + j * 8;
      b[i] = make_uint4(0, 0, 0, 0);
      if (gn < N && gk < K) b[i] = __ldg(reinterpret_cast<const uint4*>(B + (static_cast<size_t>(gn) * K + gk) * 2));
    }
  }

  // registers -> shared slot, in the layout a 128-byte-swizzled TMA copy produces
  __device__ __forceinline__ void store(uint8_t* slot) const {
    const int tid = threadIdx.x;
    const uint32_t sa = smem_u32(slot);
    const uint32_t sbb = sa + A_BYTES;
#pragma unroll
    for (int i = 0; i < A_CHUNKS; ++i) {
      const int c = tid + i * kPPThreads;
      const uint32_t addr = sa + sw128_offset(c >> 3, c & 7);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a[i].x), "r"(a[i].y), "r"(a[i].z),
                   "r"(a[i].w)
                   : "memory");
    }
#pragma unroll
    for (int i = 0; i < B_CHUNKS; ++i) {
      const int c = tid + i * kPPThreads;
      const uint32_t addr = sbb + sw128_offset(c >> 3, c & 7);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(b[i].x), "r"(b[i].y), "r"(b[i].z),
                   "r"(b[i].w)
                   : "memory");
    }
  }
};

// Epilogue for the one-tile kernels: 8 warps; warps w and w+4 share TMEM lane
// quarter w%4 and split the 64-column chunks between them.
template <int BN, bool BF16>
__device__ __forceinline__ void epilogue_8warps(uint32_t tmem, uint8_t* epi, const CUtensorMap* tmC, int M, int N,
                                                int m0, int n0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3, h = warp >> 2;
  uint8_t* buf = epi + warp * kUmmaEpiBufBytes;
  const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
  const int y = m0 + q * 32;
#pragma unroll 1
  for (int c = h; c < BN / kUmmaEpiCols; c += 2) {
    uint32_t v[64];
    load_acc_chunk(trow + c * kUmmaEpiCols, v);
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    const int x = n0 + c * kUmmaEpiCols;
    stage_and_store<BF16>(v, buf, lane, tmC, x, y, (x < N) && (y < M));
  }
  if (lane == 0) bulk_wait<0>();
}

template <int BN, bool BF16, bool PINGPONG>
__global__ void __launch_bounds__(kPPThreads, 1)
    umma_staged_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B,
                       const __grid_constant__ CUtensorMap tmC, int M, int N, int K, KernelCtl ctl) {
  constexpr int STAGE = A_BYTES + BN * BK * 2;
  constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  constexpr uint32_t IDESC = umma_idesc_f16(BF16, BM, BN);
  constexpr int NBUF = PINGPONG ? 2 : 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* epi = smem + NBUF * STAGE;
  UmmaBarriers* bar = reinterpret_cast<UmmaBarriers*>(epi + kUmmaEpiBytes);

  const int warp = threadIdx.x >> 5;
  const int m_blocks = (M + BM - 1) / BM;
  const int n_blocks = (N + BN - 1) / BN;
  int mb, nb;
  tile_coords(blockIdx.x, m_blocks, n_blocks, mb, nb);
  const int m0 = mb * BM, n0 = nb * BN;
  const int kt = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    mbar_init(&bar->mma_done[0], 1);
    mbar_init(&bar->mma_done[1], 1);
    mbar_init(&bar->drain, 1);
    bar->ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bar->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  CtaCtl* cta = &bar->ctl;
  bool ok = true;

  RegStage<BN> rs;
  if (PINGPONG) {
    // prologue: tile 0 into buffer 0
    rs.load(A, B, M, N, K, m0, n0, 0);
    rs.store(ring);
    fence_proxy_async_smem();
    __syncthreads();
    for (int kb = 0; kb < kt; ++kb) {
      const int cur = kb & 1, nxt = cur ^ 1;
      if (kb + 1 < kt) rs.load(A, B, M, N, K, m0, n0, kb + 1);   // in flight during the MMA
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + cur * STAGE);
        umma_kblock<BN>(tmem, a_addr, a_addr + A_BYTES, IDESC, kb == 0);
        umma_commit(&bar->mma_done[cur]);
      }
      if (kb + 1 < kt) {
        // buffer nxt was read by the MMAs of K step kb-1: wait for them
        if (kb >= 1)
          ok = mbar_wait(&bar->mma_done[nxt], static_cast<uint32_t>(((kb - 1) >> 1) & 1), ctl, cta,
                         kSitePingPongMma);
        if (ok) rs.store(ring + nxt * STAGE);
        fence_proxy_async_smem();
        if (!__syncthreads_and(ok ? 1 : 0)) { ok = false; break; }
      }
    }
    if (ok) {
      const int last = kt - 1;
      ok = mbar_wait(&bar->mma_done[last & 1], static_cast<uint32_t>((last >> 1) & 1), ctl, cta, kSitePingPongMma);
    }
  } else {
    for (int kb = 0; kb < kt; ++kb) {
      rs.load(A, B, M, N, K, m0, n0, kb);
      rs.store(ring);
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring);
        umma_kblock<BN>(tmem, a_addr, a_addr + A_BYTES, IDESC, kb == 0);
        umma_commit(&bar->mma_done[0]);
      }
      const bool w = mbar_wait(&bar->mma_done[0], static_cast<uint32_t>(kb & 1), ctl, cta, kSitePingPongMma);
      if (!__syncthreads_and(w ? 1 : 0)) { ok = false; break; }
    }
  }
  const int all_ok = __syncthreads_and(ok ? 1 : 0);
  if (all_ok) {
    tc_fence_after();
    epilogue_8warps<BN, BF16>(tmem, epi, &tmC, M, N, m0, n0);
  } else if (threadIdx.x == 0) {
    // MMAs may still be running: wait for all of them before TMEM is freed
    umma_commit(&bar->drain);
    CtaCtl never_abort{0};
    mbar_wait(&bar->drain, 0, ctl, &never_abort, kSiteDrain);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int BN, bool BF16, bool PAIR, bool KX = false>
cudaError_t launch_ring(LaunchArgs& a, const void** kernel) {
  using Sh = RingShape<BN, PAIR>;
  const gp_plan& p = a.plan;
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t M = a.M, N = a.N, K = a.K;
  CUtensorMap tmA, tmB, tmC;
  cudaError_t e;
  if ((e = make_tmap_2d(&tmC, a.C, dt, N, M, N * 2, kUmmaEpiCols, kUmmaEpiRows, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  if ((e = make_tmap_2d(&tmA, a.A, dt, K, M, K * 2, BK, Sh::A_ROWS, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  if ((e = make_tmap_2d(&tmB, a.B, dt, K, N, K * 2, BK, Sh::B_ROWS, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  auto k = umma_ring_kernel<BN, BF16, PAIR, KX>;
  *kernel = reinterpret_cast<const void*>(k);
  if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(Sh::THREADS);   // the plan reports the same count
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (PAIR) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = KX ? 4 : 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait() in the kernel
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, tmA, tmB, tmC, a.M, a.N, a.K, p.stages, a.ctl, a.sk);
}

template <int BN, bool BF16>
cudaError_t launch_bn(LaunchArgs& a, const void** kernel) {
  const gp_plan& p = a.plan;
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (a.variant == GP_PIPELINED) return launch_ring<BN, BF16, false>(a, kernel);
  const uint64_t M = a.M, N = a.N;
  CUtensorMap tmC;
  cudaError_t e = make_tmap_2d(&tmC, a.C, dt, N, M, N * 2, kUmmaEpiCols, kUmmaEpiRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  auto k = (a.variant == GP_PINGPONG) ? umma_staged_kernel<BN, BF16, true> : umma_staged_kernel<BN, BF16, false>;
  *kernel = reinterpret_cast<const void*>(k);
  if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
  k<<<p.grid, p.threads, p.smem_bytes, a.stream>>>(static_cast<const uint8_t*>(a.A), static_cast<const uint8_t*>(a.B),
                                                    tmC, a.M, a.N, a.K, a.ctl);
  return cudaGetLastError();
}

// INT8 on tcgen05: convert A and B to FP16 in the caller-stream workspace
// (a.conv), then run the CTA-pair chunked-accumulation kernel on them.
cudaError_t launch_i8(LaunchArgs& a, const void** kernel) {
  using Sh = RingShape<256, true>;
  const gp_plan& p = a.plan;
  const uint64_t M = a.M, N = a.N, K = a.K;
  __half* a16 = static_cast<__half*>(a.conv);
  __half* b16 = a16 + M * K;
  const int64_t na16 = static_cast<int64_t>(M * K / 16), nb16 = static_cast<int64_t>(N * K / 16);
  int64_t blocks = (na16 + nb16 + 255) / 256;
  cudaError_t e;
  if (a.conv_early) {
    // A programmatic dependent of the previous GEMM: one persistent block
    // per SM, beside that GEMM's CTAs.
    blocks = (na16 + nb16 + kEarlyConvThreads - 1) / kEarlyConvThreads;
    if (blocks > a.sm_count) blocks = a.sm_count;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kEarlyConvThreads);
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, i8_to_f16_early_kernel, static_cast<const int8_t*>(a.A), a16, na16,
                           static_cast<const int8_t*>(a.B), b16, nb16);
  } else {
    const int64_t cap = static_cast<int64_t>(a.sm_count) * 16;
    if (blocks > cap) blocks = cap;
    i8_to_f16_kernel<<<static_cast<int>(blocks), 256, 0, a.stream>>>(static_cast<const int8_t*>(a.A), a16, na16,
                                                                      static_cast<const int8_t*>(a.B), b16, nb16);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  CUtensorMap tmA, tmB, tmC;
  if ((e = make_tmap_2d(&tmC, a.C, CU_TENSOR_MAP_DATA_TYPE_INT32, N, M, N * 4, 32, kUmmaEpiRows,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  if ((e = make_tmap_2d(&tmA, a16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, M, K * 2, BK, Sh::A_ROWS,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  if ((e = make_tmap_2d(&tmB, b16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, N, K * 2, BK, Sh::B_ROWS,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  CUtensorMap tmBh;   // half items: 64 of a CTA's B rows per box
  if ((e = make_tmap_2d(&tmBh, b16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, N, K * 2, BK, Sh::B_ROWS / 2,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  auto k = umma_i8_kernel<true>;
  *kernel = reinterpret_cast<const void*>(k);
  if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlaps the conversion's tail
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // work items: the whole tiles, then two half items per tile of the N-split tail
  const int half_from = static_cast<int>(p.tiles - p.half_tiles);
  SkParams sk = a.sk;
  if (p.half_tiles > 0) sk.dp_tiles = static_cast<int32_t>(p.tiles + p.half_tiles);
  return cudaLaunchKernelEx(&cfg, k, tmA, tmB, tmC, tmBh, a.M, a.N, a.K, p.stages, a.ctl, sk, half_from);
}

// INT8 on tcgen05, the conversion overlapped inside the GEMM kernel: one launch.
cudaError_t launch_i8_overlap(LaunchArgs& a, const void** kernel) {
  using Sh = RingShape<256, true>;
  const gp_plan& p = a.plan;
  const uint64_t M = a.M, N = a.N, K = a.K;
  __half* a16 = static_cast<__half*>(a.conv);
  __half* b16 = a16 + M * K;
  CUtensorMap tmA, tmB, tmC;
  cudaError_t e;
  if ((e = make_tmap_2d(&tmC, a.C, CU_TENSOR_MAP_DATA_TYPE_INT32, N, M, N * 4, 32, kUmmaEpiRows,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  if ((e = make_tmap_2d(&tmA, a16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, M, K * 2, BK, Sh::A_ROWS,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  if ((e = make_tmap_2d(&tmB, b16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, N, K * 2, BK, Sh::B_ROWS,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  const int stg_slots = i8_overlap_staging_slots(p.stages);
  if (stg_slots < 2) return cudaErrorInvalidValue;
  CUtensorMap tmA8, tmB8;   // the int8 operands, one conversion unit (64 x 128) per box
  if ((e = make_tmap_2d(&tmA8, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, K, BK, 128, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      cudaSuccess)
    return e;
  if ((e = make_tmap_2d(&tmB8, a.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, K, BK, 128, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      cudaSuccess)
    return e;
  auto k = umma_i8_overlap_kernel;
  *kernel = reinterpret_cast<const void*>(k);
  // The warpgroups' register split is sized for a launch at exactly 128
  // registers per thread: with fewer, the epilogue's setmaxnreg.inc could not
  // be satisfied.  Refuse such a build instead of launching it.
  static std::atomic<int> launch_regs{-1};
  if (launch_regs.load() < 0) {
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, k)) != cudaSuccess) return e;
    launch_regs.store(fa.numRegs);
  }
  if (launch_regs.load() != kOvLaunchRegs) return cudaErrorInvalidConfiguration;
  if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, tmA, tmB, tmC, tmA8, tmB8, a16, b16, a.conv_ctrs, a.conv_kcap, a.conv_parity,
                            a.M, a.N, a.K, p.stages, stg_slots, a.ctl);
}

// Largest number of clusters of a pair kernel that can be resident at once.
// kind: 0 FP16 ring, 1 BF16 ring, 2 INT8 two-pass, 3 INT8 with the conversion overlapped.
// size 2: one CTA pair; size 4 (kinds 0-1, kx): two pairs splitting each 256 x 128 tile's K-loop.
cudaError_t max_clusters(int kind, int smem_bytes, int size, int* clusters, bool kx = false) {
  const void* k = kind == 3   ? reinterpret_cast<const void*>(umma_i8_overlap_kernel)
                  : kind == 2 ? reinterpret_cast<const void*>(umma_i8_kernel<true>)
                  : kx ? (kind == 1 ? reinterpret_cast<const void*>(umma_ring_kernel<128, true, true, true>)
                                    : reinterpret_cast<const void*>(umma_ring_kernel<128, false, true, true>))
                  : kind == 1 ? reinterpret_cast<const void*>(umma_ring_kernel<256, true, true, false>)
                              : reinterpret_cast<const void*>(umma_ring_kernel<256, false, true, false>);
  cudaError_t e = ensure_smem_attr(k, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(size);
  cfg.blockDim = dim3(kind == 3 ? kOvThreads : kind == 2 ? kI8Threads : RingShape<256, true>::THREADS);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, k, &cfg);
}

template <bool BF16>
cudaError_t launch_dtype(LaunchArgs& a, const void** kernel) {
  if (a.plan.cta_pair == 3) return launch_ring<128, BF16, true, true>(a, kernel);
  if (a.plan.cta_pair)
    return a.plan.bn == 128 ? launch_ring<128, BF16, true>(a, kernel) : launch_ring<256, BF16, true>(a, kernel);
  switch (a.plan.bn) {
    case 256: return launch_bn<256, BF16>(a, kernel);
    case 128: return launch_bn<128, BF16>(a, kernel);
    case 64: return launch_bn<64, BF16>(a, kernel);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_umma(LaunchArgs& a, const void** kernel) {
  return a.dtype == GP_BF16_F32ACC_BF16OUT ? launch_dtype<true>(a, kernel) : launch_dtype<false>(a, kernel);
}

cudaError_t umma_pair_capacity(int dtype, int smem_bytes, int* pairs, bool i8_overlap) {
  const int kind = dtype == GP_I8_I32 ? (i8_overlap ? 3 : 2) : (dtype == GP_BF16_F32ACC_BF16OUT ? 1 : 0);
  return max_clusters(kind, smem_bytes, 2, pairs);
}

cudaError_t umma_kx_capacity(int dtype, int smem_bytes, int* clusters) {
  return max_clusters(dtype == GP_BF16_F32ACC_BF16OUT ? 1 : 0, smem_bytes, 4, clusters, true);
}

cudaError_t launch_umma_i8(LaunchArgs& a, const void** kernel) {
  return a.i8_overlap ? launch_i8_overlap(a, kernel) : launch_i8(a, kernel);
}

}  // namespace gp
