// k_ffma.cu -- FP32 SGEMM on the CUDA cores (FFMA, no tensor cores), in the
// configuration of "CUDA Kernel Study: Pipelining", Kernel Parameters: CTA
// tile 128 x 128 x 8, 16 x 16 = 256 compute threads, 8 x 8 outputs per thread
// accumulated in registers as outer products ("Part 4 -- Pipelining and
// Occupancy", section 4.3, register tiling).  A is row-major M x K, B
// row-major K x N, C row-major M x N.
//
// The thread tile TM x TN is a template parameter (8 x 8 by default): the
// TMA ring also builds 4 x 8, 8 x 4, 8 x 16, 16 x 8 and 16 x 16, the
// register-tile sweep of "Part 4", section 4.3 (larger tiles reuse more from
// registers until the register file runs out and the compiler spills).
//
// When the tiles alone would leave SMs idle, the tiles' K-loops are dealt out
// as equal ranges to plan.grid CTAs (see FfmaWork); every data path takes the
// same ranges.
//
// Three data paths for the K-loop, sharing the shared-memory layout (A tile
// [128][8], B tile [8][128], as a TMA box copy lays them out) and the compute:
//  * ffma_ring_kernel    -- a TMA producer warp fills an S-slot ring guarded by
//                           mbarrier full/empty phases; the compute warps
//                           consume it (Case 2 with TMA + mbarrier).
//  * ffma_staged_kernel<PINGPONG=true>  -- register-staged double buffer (Case 1).
//  * ffma_staged_kernel<PINGPONG=false> -- no overlap (Background).
//
// Shared-memory access pattern (no padding or swizzle is needed): a warp's
// threads take consecutive tx and at most 32 / (128 / TN) values of ty, so an
// A read (one float4 of 4 K values of a row) touches 1-4 rows 32 bytes apart
// -- distinct 16-byte bank groups, one wavefront -- and a B read (a float4 of
// one K row) touches 128 / TN consecutive float4, the minimum number of
// wavefronts for the bytes read.  The register-staged stores write 512
// contiguous bytes per warp.
#include "gp_device.cuh"

namespace gp {
namespace {

constexpr int BM = kFfmaBM, BN = kFfmaBN, BK = kFfmaBK;
constexpr int A_FLOATS = BM * BK;          // 1024 (register-staged kernels)
constexpr int STAGE = kFfmaStageBytes;     // 8192
constexpr int SPLIT_K = kFfmaSplitK;       // K steps of one unit of a split K-loop

struct FfmaBarriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int32_t consumed;
  int32_t last;     // split K-loop: this CTA completed the tile
  CtaCtl ctl;
};
static_assert(sizeof(FfmaBarriers) <= kBarrierRegion, "barrier region too small");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void tile_coords(int tile, int m_blocks, int n_blocks, int& mb, int& nb) {
  constexpr int GM = 8;
  const int per_group = GM * n_blocks;
  const int group = tile / per_group;
  const int first_m = group * GM;
  const int gm = min(GM, m_blocks - first_m);
  const int in_group = tile - group * per_group;
  mb = first_m + in_group % gm;
  nb = in_group / gm;
}

// Thread tile TM x TN of the 128 x 128 CTA tile.  Thread (tx, ty), tx < TX,
// ty < TY, owns rows ty + TY*i (i < TM) and the float4 column groups
// g*GSTRIDE + tx*4 + {0..3} (g < NG).
template <int TM, int TN>
struct Tile {
  static constexpr int TY = BM / TM;
  static constexpr int TX = BN / TN;
  static constexpr int THREADS = TX * TY;    // compute threads
  static constexpr int WARPS = THREADS / 32;
  static constexpr int NG = TN / 4;
  static constexpr int GSTRIDE = BN / NG;
  static_assert(TN % 4 == 0 && THREADS % 32 == 0 && THREADS <= 1024, "thread tile");
};

template <int TM, int TN>
struct Acc {
  float c[TM][TN];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) c[i][j] = 0.f;
  }
};

// (c0, c1) += a * (b0, b1) as one packed FP32x2 FMA.
__device__ __forceinline__ void fma2(float& c0, float& c1, float a, float b0, float b1) {
  asm("{\n\t.reg .b64 d, x, y, z;\n\t"
      "mov.b64 x, {%2, %2};\n\t"
      "mov.b64 y, {%3, %4};\n\t"
      "mov.b64 z, {%0, %1};\n\t"
      "fma.rn.f32x2 d, x, y, z;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}\n"
      : "+f"(c0), "+f"(c1)
      : "f"(a), "f"(b0), "f"(b1));
}

// One slot of KB K steps: A as BM rows of KB, B as KB rows of BN.  (At
// KB = 32 the two A rows a warp reads at once share banks; a 128-byte TMA
// swizzle of A removed that conflict but measured 4 % slower at FP32 4096^3:
// the per-load address arithmetic costs more issue slots than it saves.)
template <int TM, int TN, int KB = BK>
__device__ __forceinline__ void ffma_kblock(const float* __restrict__ As, const float* __restrict__ Bs, int tx,
                                            int ty, Acc<TM, TN>& acc) {
  using T = Tile<TM, TN>;
#pragma unroll
  for (int kh = 0; kh < KB; kh += 4) {
    float a[TM][4];
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(As + (ty + T::TY * i) * KB + kh);
      a[i][0] = v.x; a[i][1] = v.y; a[i][2] = v.z; a[i][3] = v.w;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float b[TN];
#pragma unroll
      for (int g = 0; g < T::NG; ++g) {
        const float4 v = *reinterpret_cast<const float4*>(Bs + (kh + q) * BN + g * T::GSTRIDE + tx * 4);
        b[4 * g] = v.x; b[4 * g + 1] = v.y; b[4 * g + 2] = v.z; b[4 * g + 3] = v.w;
      }
      // Two adjacent columns per instruction: fma.rn.f32x2 is two IEEE FP32
      // FMAs (each rounded as fmaf), so the sums are bit-identical to scalar
      // FFMA, with half the instructions to issue (measured +12 % at 4096^3).
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; j += 2) fma2(acc.c[i][j], acc.c[i][j + 1], a[i][q], b[j], b[j + 1]);
    }
  }
}

template <int TM, int TN>
__device__ __forceinline__ void ffma_store(float* C, int M, int N, int m0, int n0, int tx, int ty,
                                           const Acc<TM, TN>& acc) {
  using T = Tile<TM, TN>;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int r = m0 + ty + T::TY * i;
    if (r >= M) continue;
#pragma unroll
    for (int g = 0; g < T::NG; ++g) {
      const int col = n0 + g * T::GSTRIDE + tx * 4;
      if (col < N)   // N % 4 == 0: the float4 is entirely inside
        *reinterpret_cast<float4*>(C + static_cast<size_t>(r) * N + col) =
            make_float4(acc.c[i][4 * g], acc.c[i][4 * g + 1], acc.c[i][4 * g + 2], acc.c[i][4 * g + 3]);
    }
  }
}

// Barrier of the THREADS compute threads (the ring kernel's producer warp is not in it).
template <int THREADS>
__device__ __forceinline__ void compute_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
}

// Same barrier, returning the AND of pred over the compute threads.
template <int THREADS>
__device__ __forceinline__ bool compute_bar_and(bool pred) {
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

// Work of CTA b: tile b % tiles, K steps [kb_begin, kb_end) of split b / tiles.
// Work of one CTA.  The tiles' K-loops are laid end to end (unit u: tile
// u / kt, K step u % kt) and dealt out to the G CTAs of the grid as equal
// contiguous ranges.  With G = tiles every CTA gets one whole tile; with more
// CTAs than tiles every tile's K-loop is shared by the CTAs whose ranges meet
// it, and a range (shorter than a K-loop) meets at most two tiles: its
// segment 0 (in its first tile) and segment 1.
struct FfmaWork {
  int64_t U, u, u_end;
  int kt, G;
  __device__ __forceinline__ FfmaWork(int tiles, int kt_) {
    kt = kt_;
    G = static_cast<int>(gridDim.x);
    U = static_cast<int64_t>(tiles) * kt;
    u = start(blockIdx.x);
    u_end = start(blockIdx.x + 1);
  }
  __device__ __forceinline__ int64_t start(int64_t c) const { return c * U / G; }
  // CTA whose range holds unit v
  __device__ __forceinline__ int owner(int64_t v) const { return static_cast<int>(((v + 1) * G - 1) / U); }
  // next segment of this CTA: tile, K steps [k0, k1), and its index (0 or 1) among this CTA's segments
  __device__ __forceinline__ bool next(int& tile, int& k0, int& k1, int& seg) {
    if (u >= u_end) return false;
    tile = static_cast<int>(u / kt);
    k0 = static_cast<int>(u - static_cast<int64_t>(tile) * kt);
    k1 = (u_end - u < kt - k0) ? k0 + static_cast<int>(u_end - u) : kt;
    seg = (tile == static_cast<int>(start(blockIdx.x) / kt)) ? 0 : 1;
    u += k1 - k0;
    return true;
  }
};

// Write the accumulator of one segment: to C when the segment is the whole
// K-loop, else as a partial tile (slot 2 * CTA + segment); the CTA whose
// partial completes the tile adds all of them in K order (so the sum does not
// depend on which CTA finished last) and writes C.  Called by all compute
// threads (tid < THREADS); acc is consumed (it holds the sum afterwards).
template <int TM, int TN>
__device__ __forceinline__ void ffma_finish(float* C, int M, int N, int m0, int n0, const FfmaWork& w, int tile,
                                            int seg, const FfmaSplit& ks, int tx, int ty, int tid,
                                            Acc<TM, TN>& acc, int32_t* last) {
  using T = Tile<TM, TN>;
  const int64_t t0 = static_cast<int64_t>(tile) * w.kt;
  const int c_first = w.owner(t0), c_last = w.owner(t0 + w.kt - 1);
  if (c_first == c_last) {
    ffma_store<TM, TN>(C, M, N, m0, n0, tx, ty, acc);
    return;
  }
  constexpr int TILE = BM * BN;
  float* mine = ks.workspace + (2 * static_cast<size_t>(blockIdx.x) + seg) * TILE;
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int g = 0; g < T::NG; ++g)
      __stcg(reinterpret_cast<float4*>(mine + (ty + T::TY * i) * BN + g * T::GSTRIDE + tx * 4),
             make_float4(acc.c[i][4 * g], acc.c[i][4 * g + 1], acc.c[i][4 * g + 2], acc.c[i][4 * g + 3]));
  compute_bar<T::THREADS>();
  if (tid == 0) {
    __threadfence();
    *last = (epoch_count_in(ks.counters + tile, ks.epoch) + 1u == static_cast<uint32_t>(c_last - c_first + 1)) ? 1
                                                                                                              : 0;
    __threadfence();
  }
  compute_bar<T::THREADS>();
  if (!*last) return;
  // the partials in K order, CTA c_first's segment first, summed in place of
  // this CTA's accumulator (already stored above)
  Acc<TM, TN>& tot = acc;
  for (int c = c_first; c <= c_last; ++c) {
    // the tile is segment 0 of CTA c if c's range starts in it, else its segment 1
    const int sc = (w.start(c) / w.kt == tile) ? 0 : 1;
    const float* src = ks.workspace + (2 * static_cast<size_t>(c) + sc) * TILE;
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int g = 0; g < T::NG; ++g) {
        const float4 p = __ldcg(reinterpret_cast<const float4*>(src + (ty + T::TY * i) * BN + g * T::GSTRIDE + tx * 4));
        float* d = &tot.c[i][4 * g];
        if (c == c_first) {
          d[0] = p.x;
          d[1] = p.y;
          d[2] = p.z;
          d[3] = p.w;
        } else {
          d[0] += p.x;
          d[1] += p.y;
          d[2] += p.z;
          d[3] += p.w;
        }
      }
  }
  ffma_store<TM, TN>(C, M, N, m0, n0, tx, ty, tot);
}

// ---------------------------------------------------------------------------
// TMA ring: compute warps + 1 producer warp, one (tile, K split) per CTA
// ---------------------------------------------------------------------------
// SPLIT: some tile's K-loop is shared by several CTAs (else each CTA runs one
// whole tile and stores it directly; a separate instantiation keeps the
// fix-up code out of that kernel).
template <int TM, int TN, bool SPLIT, int RBK>
__global__ void __launch_bounds__(Tile<TM, TN>::THREADS + 32, 1)
    ffma_ring_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     float* __restrict__ C, int M, int N, int K, int stages, KernelCtl ctl, FfmaSplit ks) {
  using T = Tile<TM, TN>;
  constexpr int RA_FLOATS = BM * RBK;
  constexpr int RSTAGE = (BM * RBK + RBK * BN) * 4;
  constexpr int R = SPLIT_K / RBK;   // slots per unit of a split K-loop
  static_assert(SPLIT_K % RBK == 0, "split unit");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align1024(smem_raw);
  FfmaBarriers* bar = reinterpret_cast<FfmaBarriers*>(ring + stages * RSTAGE);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_blocks = (M + BM - 1) / BM, n_blocks = (N + BN - 1) / BN;
  const int kt = (K + RBK - 1) / RBK;
  const int tiles = m_blocks * n_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar->full[s], 1);
      mbar_init(&bar->empty[s], T::WARPS);
    }
    bar->ctl.abort = 0;
    bar->consumed = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent: the set-up above overlaps the
  // previous kernel's tail.  The producer reads A and B only after that
  // kernel has completed (or at once, when the caller promised that nothing
  // in flight writes them); the compute warps write C and the split
  // workspace only after it has completed.
  pdl_launch_dependents();
  CtaCtl* cta = &bar->ctl;
  int issued = 0;
  FfmaWork wk(tiles, (K + SPLIT_K - 1) / SPLIT_K);
  int tile, u0, u1, seg;

  if (warp == T::WARPS) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int s = 0;
      uint32_t ph = 0;
      const bool last_cta = blockIdx.x == gridDim.x - 1;
      if (!ctl.inputs_ready) pdl_wait();
      bool ok = true;
      while (ok && wk.next(tile, u0, u1, seg)) {
        int mb, nb;
        tile_coords(tile, m_blocks, n_blocks, mb, nb);
        const int k0 = u0 * R, k1 = min(u1 * R, kt);
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(&bar->empty[s], ph ^ 1u, ctl, cta, kSiteProducerEmpty)) { ok = false; break; }
          if (!(ctl.inject_lost_load && last_cta && wk.u >= wk.u_end && kb == k1 - 1)) {
            uint8_t* slot = ring + s * RSTAGE;
            mbar_arrive_expect_tx(&bar->full[s], RSTAGE);
            tma_load_2d(smem_u32(slot), &tmA, &bar->full[s], kb * RBK, mb * BM);
            tma_load_2d(smem_u32(slot + RA_FLOATS * 4), &tmB, &bar->full[s], nb * BN, kb * RBK);
            ++issued;
          }
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else {
    const int tx = threadIdx.x % T::TX, ty = threadIdx.x / T::TX;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    int consumed = 0;
    bool waited = false;
    if (!ctl.inputs_ready) {
      // The producer's loads start only after the previous kernel has completed,
      // so start the bounded waits on full slots only then too: a long-running
      // predecessor must not use up their time limit.
      pdl_wait();
      waited = true;
    }
    while (ok && wk.next(tile, u0, u1, seg)) {
      int mb, nb;
      tile_coords(tile, m_blocks, n_blocks, mb, nb);
      const int k0 = u0 * R, k1 = min(u1 * R, kt);
      Acc<TM, TN> acc;
      acc.zero();
      for (int kb = k0; kb < k1; ++kb) {
        const bool w = mbar_wait(&bar->full[s], ph, ctl, cta, kSiteConsumerFull);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        const float* As = reinterpret_cast<const float*>(ring + s * RSTAGE);
        ffma_kblock<TM, TN, RBK>(As, As + RA_FLOATS, tx, ty, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->empty[s]);
        ++consumed;
        if (++s == stages) { s = 0; ph ^= 1u; }
      }
      // one decision for all compute warps: a timed-out warp must not leave the others at a barrier
      ok = compute_bar_and<T::THREADS>(ok);
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      if (ok) {
        if (SPLIT)
          ffma_finish<TM, TN>(C, M, N, mb * BM, nb * BN, wk, tile, seg, ks, tx, ty, threadIdx.x, acc, &bar->last);
        else
          ffma_store<TM, TN>(C, M, N, mb * BM, nb * BN, tx, ty, acc);
      }
    }
    if (threadIdx.x == 0) bar->consumed = consumed;
  }

  __syncthreads();
  if (cta->abort && warp == T::WARPS && lane == 0) {
    CtaCtl never_abort{0};
    for (int i = bar->consumed; i < issued; ++i)
      mbar_wait(&bar->full[i % stages], static_cast<uint32_t>((i / stages) & 1), ctl, &never_abort, kSiteDrain);
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// register-staged ping-pong / no-overlap (the 8 x 8 thread tile, 256 threads)
// ---------------------------------------------------------------------------
constexpr int kStagedThreads = Tile<8, 8>::THREADS;

struct RegStage {
  float4 a, b;
  // A: thread t loads row t/2, k-quad t%2; B: row t/32, column quad t%32
  __device__ __forceinline__ void load(const float* A, const float* B, int M, int N, int K, int m0, int n0, int kb) {
    const int t = threadIdx.x;
    const int k0 = kb * BK;
    const int gm = m0 + (t >> 1), gk = k0 + (t & 1) * 4;
    a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gm < M && gk < K) a = __ldg(reinterpret_cast<const float4*>(A + static_cast<size_t>(gm) * K + gk));
    const int bk = k0 + (t >> 5), bn = n0 + (t & 31) * 4;
    b = make_float4(0.f, 0.f, 0.f, 0.f);
    if (bk < K && bn < N) b = __ldg(reinterpret_cast<const float4*>(B + static_cast<size_t>(bk) * N + bn));
  }
  __device__ __forceinline__ void store(uint8_t* slot) const {
    const int t = threadIdx.x;
    float* As = reinterpret_cast<float*>(slot);
    float* Bs = As + A_FLOATS;
    *reinterpret_cast<float4*>(As + (t >> 1) * BK + (t & 1) * 4) = a;
    *reinterpret_cast<float4*>(Bs + (t >> 5) * BN + (t & 31) * 4) = b;
  }
};

template <bool PINGPONG>
__global__ void __launch_bounds__(kStagedThreads, 1)
    ffma_staged_kernel(const float* __restrict__ A, const float* __restrict__ B, float* __restrict__ C, int M, int N,
                       int K, FfmaSplit ks) {
  using T = Tile<8, 8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int32_t last;
  uint8_t* ring = align1024(smem_raw);
  const int m_blocks = (M + BM - 1) / BM, n_blocks = (N + BN - 1) / BN;
  const int kt = (K + BK - 1) / BK;
  const int tx = threadIdx.x % T::TX, ty = threadIdx.x / T::TX;
  // A K-loop shared by several CTAs is cut every SPLIT_K K steps, as in the
  // ring, so every variant adds the same partial sums: a unit is R tiles here.
  constexpr int R = SPLIT_K / BK;
  static_assert(SPLIT_K % BK == 0, "split unit");
  FfmaWork wk(m_blocks * n_blocks, (K + SPLIT_K - 1) / SPLIT_K);
  int tile, u0, u1, seg;
  while (wk.next(tile, u0, u1, seg)) {
    int mb, nb;
    tile_coords(tile, m_blocks, n_blocks, mb, nb);
    const int m0 = mb * BM, n0 = nb * BN;
    const int k0 = u0 * R, k1 = min(u1 * R, kt);
    Acc<8, 8> acc;
    acc.zero();
    RegStage rs;
    if (PINGPONG) {
      rs.load(A, B, M, N, K, m0, n0, k0);
      rs.store(ring);
      __syncthreads();
      for (int kb = k0; kb < k1; ++kb) {
        const int cur = (kb - k0) & 1;
        if (kb + 1 < k1) rs.load(A, B, M, N, K, m0, n0, kb + 1);   // in flight during the compute
        const float* As = reinterpret_cast<const float*>(ring + cur * STAGE);
        ffma_kblock<8, 8>(As, As + A_FLOATS, tx, ty, acc);
        if (kb + 1 < k1) rs.store(ring + (cur ^ 1) * STAGE);   // last read in iteration kb-1
        __syncthreads();
      }
    } else {
      for (int kb = k0; kb < k1; ++kb) {
        rs.load(A, B, M, N, K, m0, n0, kb);
        rs.store(ring);
        __syncthreads();
        const float* As = reinterpret_cast<const float*>(ring);
        ffma_kblock<8, 8>(As, As + A_FLOATS, tx, ty, acc);
        __syncthreads();
      }
    }
    ffma_finish<8, 8>(C, M, N, m0, n0, wk, tile, seg, ks, tx, ty, threadIdx.x, acc, &last);
  }
}

template <int TM, int TN>
cudaError_t launch_ring_tile(LaunchArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB, const void** kernel) {
  const gp_plan& p = a.plan;
  auto k = p.bk == 32 ? (p.k_splits > 1 ? ffma_ring_kernel<TM, TN, true, 32> : ffma_ring_kernel<TM, TN, false, 32>)
                      : (p.k_splits > 1 ? ffma_ring_kernel<TM, TN, true, 16> : ffma_ring_kernel<TM, TN, false, 16>);
  *kernel = reinterpret_cast<const void*>(k);
  cudaError_t e = ensure_smem_attr(*kernel, p.smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(Tile<TM, TN>::THREADS + 32);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait() in the kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, tmA, tmB, static_cast<float*>(a.C), a.M, a.N, a.K, p.stages, a.ctl, a.ks);
}

}  // namespace

// Compute threads of the FFMA ring for a thread tile (0 if that tile is not built).
int ffma_ring_compute_threads(int tm, int tn) {
  switch (tm * 100 + tn) {
    case 408: case 804: case 808: case 816: case 1608: case 1616: return (BM / tm) * (BN / tn);
    default: return 0;
  }
}

cudaError_t launch_ffma(LaunchArgs& a, const void** kernel) {
  gp_plan& p = a.plan;
  cudaError_t e;
  if (a.variant == GP_PIPELINED) {
    CUtensorMap tmA, tmB;
    const uint64_t M = a.M, N = a.N, K = a.K;
    const int rbk = p.bk;   // K steps per ring slot: 32, or 16 for 7-8 slots
    if (rbk != 32 && rbk != 16) return cudaErrorInvalidValue;
    if ((e = make_tmap_2d(&tmA, a.A, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, K, M, K * 4, rbk, BM,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
      return e;
    if ((e = make_tmap_2d(&tmB, a.B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, N, K, N * 4, BN, rbk,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
      return e;
    switch (a.ffma_tm * 100 + a.ffma_tn) {
      case 408: return launch_ring_tile<4, 8>(a, tmA, tmB, kernel);
      case 804: return launch_ring_tile<8, 4>(a, tmA, tmB, kernel);
      case 808: return launch_ring_tile<8, 8>(a, tmA, tmB, kernel);
      case 816: return launch_ring_tile<8, 16>(a, tmA, tmB, kernel);
      case 1608: return launch_ring_tile<16, 8>(a, tmA, tmB, kernel);
      case 1616: return launch_ring_tile<16, 16>(a, tmA, tmB, kernel);
      default: return cudaErrorInvalidValue;
    }
  }
  auto k = (a.variant == GP_PINGPONG) ? ffma_staged_kernel<true> : ffma_staged_kernel<false>;
  *kernel = reinterpret_cast<const void*>(k);
  if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
  k<<<p.grid, kStagedThreads, p.smem_bytes, a.stream>>>(static_cast<const float*>(a.A), static_cast<const float*>(a.B),
                                                        static_cast<float*>(a.C), a.M, a.N, a.K, a.ks);
  return cudaGetLastError();
}

}  // namespace gp
