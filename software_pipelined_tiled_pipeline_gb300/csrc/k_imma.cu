// k_imma.cu -- INT8 x INT8 -> INT32 GEMM with warp-level IMMA
// (mma.sync.m16n8k32.s32.s8.s8.s32).  sm_103a has no integer kind of
// tcgen05.mma, so the INT8 consumers are warps; the K-loop data paths are the
// same three as for the other element types:
//
//  * imma_ring_kernel  -- the main path.  Persistent and warp-specialised: a
//    TMA producer warp fills an S-slot shared-memory ring (mbarrier full /
//    empty phases); eight consumer warps run ldmatrix + IMMA on each slot and
//    release it with one arrival per warp.  While consumers write one tile's
//    result the producer is already filling the ring for the next tile.
//    ("CUDA Kernel Study: Pipelining", Case 2, with TMA + mbarrier in place of
//    cp.async commit/wait groups.)
//  * imma_staged_kernel<PINGPONG=true> -- register-staged double buffer
//    (Case 1; "pipeline-gpu-kernel" Step 3, LDG-register variant): the global
//    loads of tile k+1 are in flight in registers while the warps compute on
//    tile k, then the registers go to the other buffer and one barrier
//    separates the iterations.
//  * imma_staged_kernel<PINGPONG=false> -- load, barrier, compute, barrier.
//
// Shared tiles are K-major 128-byte rows stored with the TMA 128-byte swizzle
// in every variant, so ldmatrix reads are conflict-free and the compute code
// is identical.  Integer sums wrap modulo 2^32 like the definition.
#include "gp_device.cuh"

namespace gp {
namespace {

constexpr int BM = kImmaBM;   // 128
constexpr int BK = kImmaBK;   // 128 int8 = 128 bytes per row
constexpr int A_BYTES = BM * BK;
constexpr int kConsumerWarps = 8;   // 2 (M) x 4 (N)

struct ImmaBarriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int32_t consumed;
  CtaCtl ctl;
};
static_assert(sizeof(ImmaBarriers) <= kBarrierRegion, "barrier region too small");

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

// Accumulators of one consumer warp: warp tile 64 x (BN/4): 4 m16 tiles x NT n8 tiles.
template <int BN>
struct WarpAcc {
  static constexpr int WN = BN / 4;
  static constexpr int NT = WN / 8;
  int32_t c[4][NT][4];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int r = 0; r < 4; ++r) c[i][j][r] = 0;
  }
};

// One 128-wide K step of a warp: 4 k32 sub-steps, ldmatrix fragments from the
// swizzled slot (sA: 128 rows, sB: BN rows, 128 bytes each).
template <int BN>
__device__ __forceinline__ void imma_kblock(uint32_t sA, uint32_t sB, int wm, int wn, int lane, WarpAcc<BN>& acc) {
  constexpr int WN = WarpAcc<BN>::WN;
  constexpr int NT = WarpAcc<BN>::NT;
#pragma unroll
  for (int ks = 0; ks < BK / 32; ++ks) {
    uint32_t a[4][4];
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
      // matrices: (rows 0-7, k 0-15) (rows 8-15, k 0-15) (rows 0-7, k 16-31) (rows 8-15, k 16-31)
      const uint32_t row = wm * 64 + mi * 16 + (lane & 15);
      const uint32_t chunk = ks * 2 + (lane >> 4);
      ldmatrix_x4(sA + sw128_offset(row, chunk), a[mi][0], a[mi][1], a[mi][2], a[mi][3]);
    }
    uint32_t b[NT][2];
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      // matrices: (n 0-7, k 0-15) (n 0-7, k 16-31) (n 8-15, k 0-15) (n 8-15, k 16-31)
      const uint32_t nrow = wn * WN + np * 16 + ((lane >> 4) & 1) * 8 + (lane & 7);
      const uint32_t chunk = ks * 2 + ((lane >> 3) & 1);
      ldmatrix_x4(sB + sw128_offset(nrow, chunk), b[2 * np][0], b[2 * np][1], b[2 * np + 1][0], b[2 * np + 1][1]);
    }
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
      for (int ni = 0; ni < NT; ++ni) mma_s8_16832(acc.c[mi][ni], a[mi], b[ni][0], b[ni][1]);
  }
}

// INT32 results of one warp straight from registers: each quad of lanes
// writes 8 contiguous bytes of a row, so every 32-byte sector is filled.
template <int BN>
__device__ __forceinline__ void imma_store(int32_t* C, int M, int N, int m0, int n0, int wm, int wn, int lane,
                                           const WarpAcc<BN>& acc) {
  constexpr int WN = WarpAcc<BN>::WN;
  constexpr int NT = WarpAcc<BN>::NT;
#pragma unroll
  for (int mi = 0; mi < 4; ++mi) {
    const int r0 = m0 + wm * 64 + mi * 16 + (lane >> 2);
#pragma unroll
    for (int ni = 0; ni < NT; ++ni) {
      const int col = n0 + wn * WN + ni * 8 + (lane & 3) * 2;
      if (col < N) {   // N % 4 == 0 and col even: col + 1 < N as well
        if (r0 < M)
          *reinterpret_cast<int2*>(C + static_cast<size_t>(r0) * N + col) =
              make_int2(acc.c[mi][ni][0], acc.c[mi][ni][1]);
        if (r0 + 8 < M)
          *reinterpret_cast<int2*>(C + static_cast<size_t>(r0 + 8) * N + col) =
              make_int2(acc.c[mi][ni][2], acc.c[mi][ni][3]);
      }
    }
  }
}

// Every lane waits (each acquires the phase); the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const KernelCtl& ctl, CtaCtl* cta,
                                          uint32_t site) {
  const bool ok = mbar_wait(bar, parity, ctl, cta, site);
  return __all_sync(0xffffffffu, ok) != 0;
}

// ---------------------------------------------------------------------------
// main path: persistent TMA ring, 8 consumer warps + 1 producer warp
// ---------------------------------------------------------------------------
template <int BN>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 1)
    imma_ring_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     int32_t* __restrict__ C, int M, int N, int K, int stages, KernelCtl ctl) {
  constexpr int STAGE = A_BYTES + BN * BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align1024(smem_raw);
  ImmaBarriers* bar = reinterpret_cast<ImmaBarriers*>(ring + stages * STAGE);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_blocks = (M + BM - 1) / BM, n_blocks = (N + BN - 1) / BN;
  const int tiles = m_blocks * n_blocks;
  const int kt = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar->full[s], 1);
      mbar_init(&bar->empty[s], kConsumerWarps);
    }
    bar->ctl.abort = 0;
    bar->consumed = 0;
    fence_mbar_init();
  }
  __syncthreads();
  CtaCtl* cta = &bar->ctl;
  int issued = 0;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int s = 0;
      uint32_t ph = 0;
      for (int tile = blockIdx.x; tile < tiles && !cta->abort; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, m_blocks, n_blocks, mb, nb);
        for (int kb = 0; kb < kt; ++kb) {
          if (!mbar_wait(&bar->empty[s], ph ^ 1u, ctl, cta, kSiteProducerEmpty)) goto producer_done;
          const bool drop = ctl.inject_lost_load && tile == tiles - 1 && kb == kt - 1;
          if (!drop) {
            uint8_t* slot = ring + s * STAGE;
            mbar_arrive_expect_tx(&bar->full[s], STAGE);
            tma_load_2d(smem_u32(slot), &tmA, &bar->full[s], kb * BK, mb * BM);
            tma_load_2d(smem_u32(slot + A_BYTES), &tmB, &bar->full[s], kb * BK, nb * BN);
            ++issued;
          }
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
    producer_done:;
    }
  } else {
    // ---------------- consumers ----------------
    const int wm = warp >> 2, wn = warp & 3;
    int s = 0;
    uint32_t ph = 0;
    int consumed = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, m_blocks, n_blocks, mb, nb);
      WarpAcc<BN> acc;
      acc.zero();
      for (int kb = 0; kb < kt; ++kb) {
        if (!warp_wait(&bar->full[s], ph, ctl, cta, kSiteConsumerFull)) { ok = false; break; }
        const uint32_t sa = smem_u32(ring + s * STAGE);
        imma_kblock<BN>(sa, sa + A_BYTES, wm, wn, lane, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->empty[s]);
        ++consumed;
        if (++s == stages) { s = 0; ph ^= 1u; }
      }
      if (ok) imma_store<BN>(C, M, N, mb * BM, nb * BN, wm, wn, lane, acc);
    }
    if (warp == 0 && lane == 0) bar->consumed = consumed;
  }

  __syncthreads();
  if (cta->abort && warp == kConsumerWarps && lane == 0) {
    // wait for loads still landing in shared memory before the CTA exits
    CtaCtl never_abort{0};
    for (int i = bar->consumed; i < issued; ++i)
      mbar_wait(&bar->full[i % stages], static_cast<uint32_t>((i / stages) & 1), ctl, &never_abort, kSiteDrain);
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// register-staged ping-pong / no-overlap (256 threads = the 8 consumer warps)
// ---------------------------------------------------------------------------
constexpr int kPPThreads = kConsumerWarps * 32;

template <int BN>
struct RegStage {
  static constexpr int A_CHUNKS = BM * 8 / kPPThreads;   // 4
  static constexpr int B_CHUNKS = BN * 8 / kPPThreads;   // BN / 32
  uint4 a[A_CHUNKS];
  uint4 b[B_CHUNKS];

  __device__ __forceinline__ void load(const int8_t* A, const int8_t* B, int M, int N, int K, int m0, int n0,
                                       int kb) {
    const int tid = threadIdx.x;
    const int k0 = kb * BK;
#pragma unroll
    for (int i = 0; i < A_CHUNKS; ++i) {
      const int c = tid + i * kPPThreads;
      const int gm = m0 + (c >> 3), gk = k0 + (c & 7) * 16;
      a[i] = make_uint4(0, 0, 0, 0);
      if (gm < M && gk < K) a[i] = __ldg(reinterpret_cast<const uint4*>(A + static_cast<size_t>(gm) * K + gk));
    }
#pragma unroll
    for (int i = 0; i < B_CHUNKS; ++i) {
      const int c = tid + i * kPPThreads;
      const int gn = n0 + (c >> 3), gk = k0 + (c & 7) * 16;
      b[i] = make_uint4(0, 0, 0, 0);
      if (gn < N && gk < K) b[i] = __ldg(reinterpret_cast<const uint4*>(B + static_cast<size_t>(gn) * K + gk));
    }
  }

  __device__ __forceinline__ void store(uint8_t* slot) const {
    const int tid = threadIdx.x;
    const uint32_t sa = smem_u32(slot), sb = sa + A_BYTES;
#pragma unroll
    for (int i = 0; i < A_CHUNKS; ++i) {
      const int c = tid + i * kPPThreads;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sa + sw128_offset(c >> 3, c & 7)), "r"(a[i].x),
                   "r"(a[i].y), "r"(a[i].z), "r"(a[i].w)
                   : "memory");
    }
#pragma unroll
    for (int i = 0; i < B_CHUNKS; ++i) {
      const int c = tid + i * kPPThreads;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sb + sw128_offset(c >> 3, c & 7)), "r"(b[i].x),
                   "r"(b[i].y), "r"(b[i].z), "r"(b[i].w)
                   : "memory");
    }
  }
};

template <int BN, bool PINGPONG>
__global__ void __launch_bounds__(kPPThreads, 1)
    imma_staged_kernel(const int8_t* __restrict__ A, const int8_t* __restrict__ B, int32_t* __restrict__ C, int M,
                       int N, int K) {
  constexpr int STAGE = A_BYTES + BN * BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align1024(smem_raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp >> 2, wn = warp & 3;
  const int m_blocks = (M + BM - 1) / BM, n_blocks = (N + BN - 1) / BN;
  int mb, nb;
  tile_coords(blockIdx.x, m_blocks, n_blocks, mb, nb);
  const int m0 = mb * BM, n0 = nb * BN;
  const int kt = (K + BK - 1) / BK;

  WarpAcc<BN> acc;
  acc.zero();
  RegStage<BN> rs;
  if (PINGPONG) {
    rs.load(A, B, M, N, K, m0, n0, 0);
    rs.store(ring);
    __syncthreads();
    for (int kb = 0; kb < kt; ++kb) {
      const int cur = kb & 1;
      if (kb + 1 < kt) rs.load(A, B, M, N, K, m0, n0, kb + 1);   // in flight during the compute
      const uint32_t sa = smem_u32(ring + cur * STAGE);
      imma_kblock<BN>(sa, sa + A_BYTES, wm, wn, lane, acc);
      // the other buffer was last read in iteration kb-1, which every thread
      // finished before the barrier that ended it
      if (kb + 1 < kt) rs.store(ring + (cur ^ 1) * STAGE);
      __syncthreads();
    }
  } else {
    for (int kb = 0; kb < kt; ++kb) {
      rs.load(A, B, M, N, K, m0, n0, kb);
      rs.store(ring);
      __syncthreads();
      const uint32_t sa = smem_u32(ring);
      imma_kblock<BN>(sa, sa + A_BYTES, wm, wn, lane, acc);
      __syncthreads();
    }
  }
  imma_store<BN>(C, M, N, m0, n0, wm, wn, lane, acc);
}

template <int BN>
cudaError_t launch_bn(LaunchArgs& a, const void** kernel) {
  gp_plan& p = a.plan;
  cudaError_t e;
  if (a.variant == GP_PIPELINED) {
    CUtensorMap tmA, tmB;
    const uint64_t M = a.M, N = a.N, K = a.K;
    if ((e = make_tmap_2d(&tmA, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        cudaSuccess)
      return e;
    if ((e = make_tmap_2d(&tmB, a.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, K, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        cudaSuccess)
      return e;
    auto k = imma_ring_kernel<BN>;
    *kernel = reinterpret_cast<const void*>(k);
    if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
    int occ = 1;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, p.threads, p.smem_bytes)) != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    const int64_t cap = a.one_tile ? p.tiles : static_cast<int64_t>(a.sm_count) * occ;
    p.grid = static_cast<int32_t>(p.tiles < cap ? p.tiles : cap);
    k<<<p.grid, p.threads, p.smem_bytes, a.stream>>>(tmA, tmB, static_cast<int32_t*>(a.C), a.M, a.N, a.K, p.stages,
                                                      a.ctl);
  } else {
    auto k = (a.variant == GP_PINGPONG) ? imma_staged_kernel<BN, true> : imma_staged_kernel<BN, false>;
    *kernel = reinterpret_cast<const void*>(k);
    if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
    k<<<p.grid, p.threads, p.smem_bytes, a.stream>>>(static_cast<const int8_t*>(a.A), static_cast<const int8_t*>(a.B),
                                                      static_cast<int32_t*>(a.C), a.M, a.N, a.K);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_imma(LaunchArgs& a, const void** kernel) {
  switch (a.plan.bn) {
    case 128: return launch_bn<128>(a, kernel);
    case 64: return launch_bn<64>(a, kernel);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gp
