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
//    overlaps the K-loop of the next.  This is the S-stage ring of
//    "CUDA Kernel Study: Pipelining", Case 2 (prologue fills S slots, the
//    steady state refills the slot just consumed, the tail drains), with TMA
//    completion bytes on an mbarrier in place of cp.async commit/wait groups.
//
//  * umma_pingpong_kernel -- the register-staged double buffer of Case 1 /
//    "pipeline-gpu-kernel" Step 3 (LDG-register variant): global loads of tile
//    k+1 into registers are in flight while the tensor core consumes tile k
//    from one shared buffer; the registers are then stored to the other
//    buffer.  The "compute finished reading" barrier before that store is the
//    tcgen05.commit of the previous tile's MMAs.
//
//  * umma_nopipe_kernel -- load, synchronise, compute, wait (Background).
//
// All three use the same tile shape, shared-memory layout (K-major tiles of
// 128-byte rows with the 128-byte swizzle), MMA sequence and epilogue, so
// they differ only in how tiles reach shared memory.
#include "gp_device.cuh"

namespace gp {
namespace {

constexpr int BM = kUmmaBM;   // 128
constexpr int BK = kUmmaBK;   // 64 elements = 128 bytes per row
constexpr int A_BYTES = BM * BK * 2;
constexpr int UMMA_K = 16;    // K of one kind::f16 instruction

struct UmmaBarriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t consumed_hi;        // k-blocks consumed by the MMA thread (low 31 bits)
  CtaCtl ctl;
};
static_assert(sizeof(UmmaBarriers) <= kBarrierRegion, "barrier region too small");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Grouped raster: GM consecutive M-blocks share each N-block sweep, so the
// CTAs resident at one time reuse A and B tiles through L2.
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
__device__ __forceinline__ void stage_and_store(const uint32_t (&v)[64], uint8_t* buf, int lane,
                                                const CUtensorMap* tmap_c, int x, int y, bool in_bounds) {
  uint32_t p[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) p[i] = pack2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), BF16);
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

__device__ __forceinline__ void load_acc_chunk(uint32_t taddr, uint32_t (&v)[64]) {
  uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
  uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
  tmem_ld_32x32b_x32(taddr, lo);
  tmem_ld_32x32b_x32(taddr + 32, hi);
  tmem_wait_ld();
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
template <int BN, bool BF16>
__global__ void __launch_bounds__(192, 1)
    umma_ring_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, int M, int N, int K, int stages, KernelCtl ctl) {
  constexpr int STAGE = A_BYTES + BN * BK * 2;
  constexpr uint32_t TMEM_COLS = 2 * BN;
  constexpr uint32_t IDESC = umma_idesc_f16(BF16, BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* epi = smem + stages * STAGE;
  UmmaBarriers* bar = reinterpret_cast<UmmaBarriers*>(epi + kUmmaEpiBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_blocks = (M + BM - 1) / BM;
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
      mbar_init(&bar->acc_empty[a], kUmmaEpiWarps);
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
    tmem_alloc(&bar->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  CtaCtl* cta = &bar->ctl;
  int issued = 0;  // producer only

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
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
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int consumed = 0;
      int t = 0;
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++t) {
        const int a = t & 1;
        if (!mbar_wait(&bar->acc_empty[a], ((t >> 1) & 1) ^ 1u, ctl, cta, kSiteMmaAccEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem + a * BN;
        bool ok = true;
        for (int kb = 0; kb < kt; ++kb) {
          if (!mbar_wait(&bar->full[s], ph, ctl, cta, kSiteConsumerFull)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(ring + s * STAGE);
          umma_kblock<BN>(d, a_addr, a_addr + A_BYTES, IDESC, kb == 0);
          umma_commit(&bar->empty[s]);   // slot s is free once these MMAs have read it
          ++consumed;
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&bar->acc_full[a]);  // accumulator a complete
      }
      bar->consumed_hi = consumed;
      // every MMA issued by this thread has completed once drain fires
      umma_commit(&bar->drain);
      KernelCtl c2 = ctl;
      CtaCtl never_abort{0};
      mbar_wait(&bar->drain, 0, c2, &never_abort, kSiteDrain);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int e = warp - 2;
    uint8_t* my_stage = epi + e * 2 * kUmmaEpiBufBytes;
    int sb = 0;
    int t = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++t) {
      int mb, nb;
      tile_coords(tile, m_blocks, n_blocks, mb, nb);
      const int a = t & 1;
      uint32_t ok = 1;
      if (lane == 0) ok = mbar_wait(&bar->acc_full[a], (t >> 1) & 1, ctl, cta, kSiteEpilogueAccFull) ? 1u : 0u;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * BN;
      const int y = mb * BM + q * 32;
#pragma unroll 1
      for (int c = 0; c < BN / kUmmaEpiCols; ++c) {
        uint32_t v[64];
        load_acc_chunk(trow + c * kUmmaEpiCols, v);
        if (c == BN / kUmmaEpiCols - 1) {
          // all of accumulator a is in registers: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar->acc_empty[a]);
        }
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        const int x = nb * BN + c * kUmmaEpiCols;
        stage_and_store<BF16>(v, my_stage + sb * kUmmaEpiBufBytes, lane, &tmC, x, y, (x < N) && (y < M));
        sb ^= 1;
      }
    }
    if (lane == 0) bulk_wait<0>();
  }

  __syncthreads();
  if (cta->abort && warp == 0 && lane == 0) {
    // loads still in flight land in shared memory: wait for them before exit
    CtaCtl never_abort{0};
    const int done = bar->consumed_hi;
    for (int i = done; i < issued; ++i) {
      const int s = i % stages;
      mbar_wait(&bar->full[s], static_cast<uint32_t>((i / stages) & 1), ctl, &never_abort, kSiteDrain);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
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

template <int BN, bool BF16>
cudaError_t launch_bn(LaunchArgs& a, const void** kernel) {
  const gp_plan& p = a.plan;
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t M = a.M, N = a.N, K = a.K;
  CUtensorMap tmC;
  cudaError_t e = make_tmap_2d(&tmC, a.C, dt, N, M, N * 2, kUmmaEpiCols, kUmmaEpiRows,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  if (a.variant == GP_PIPELINED) {
    CUtensorMap tmA, tmB;
    if ((e = make_tmap_2d(&tmA, a.A, dt, K, M, K * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&tmB, a.B, dt, K, N, K * 2, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
    auto k = umma_ring_kernel<BN, BF16>;
    *kernel = reinterpret_cast<const void*>(k);
    if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
    k<<<p.grid, p.threads, p.smem_bytes, a.stream>>>(tmA, tmB, tmC, a.M, a.N, a.K, p.stages, a.ctl);
  } else {
    auto k = (a.variant == GP_PINGPONG) ? umma_staged_kernel<BN, BF16, true> : umma_staged_kernel<BN, BF16, false>;
    *kernel = reinterpret_cast<const void*>(k);
    if ((e = ensure_smem_attr(*kernel, p.smem_bytes)) != cudaSuccess) return e;
    k<<<p.grid, p.threads, p.smem_bytes, a.stream>>>(static_cast<const uint8_t*>(a.A),
                                                      static_cast<const uint8_t*>(a.B), tmC, a.M, a.N, a.K, a.ctl);
  }
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_dtype(LaunchArgs& a, const void** kernel) {
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

}  // namespace gp
