// gemm_bf16.cu - persistent grouped GEMMs of the expert block on the
// 5th-generation tensor cores (tcgen05) of sm_103a.
//
// Structure (one CTA per SM, 6 warps):
//   warp 0      TMA producer: streams the A tile (128 routed rows x 64 of K)
//               and the B tile (64 of K x 256 weight columns) of every
//               k-block into a ring of `stages` shared-memory slots.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=256,
//               K=16) on each slot and releases it with tcgen05.commit;
//               accumulates a tile in one of two TMEM buffers (2 x 256
//               columns) so that the epilogue of tile i overlaps tile i+1.
//   warps 2-5   epilogue: tcgen05.ld the accumulator, apply SwiGLU (fc1) or
//               round (fc2), store bf16 rows.
// This is the in-kernel counterpart of the MC2 ring of "MC2 通算融合架构总览"
// (sections 3-4): the producer's TMA loads stand where the AIV's UDMA puts
// stood, the mbarrier pair full/empty where the CrossCore set/wait flags
// stood, and slot = k-block mod stages as bufferId = mLoopIdx mod bufferSize.
//
// Tiles: expert e owns rows [off_al[e], off_al[e+1]) of the permuted
// activations, a multiple of 128 (padded), i.e. (off_al[e+1]-off_al[e])/128
// M tiles, times N/bn N tiles. The persistent scheduler numbers the tiles of
// all experts consecutively (M fastest, so CTAs that run at the same time
// share one weight tile through L2) and CTA b takes tiles b, b+grid, ...
// Experts without rows own no tile. Counts never leave the device.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int BK = 64;                         // k-block (128 bytes of bf16)
constexpr int kABytes = kTileM * BK * 2;       // 16 KB
constexpr int kBBox = 64 * BK * 2;             // 8 KB: 64 columns x 64 of K
constexpr int kStageBytes = kABytes + 4 * kBBox;  // 48 KB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kDrainNs = 1000000000ull;

struct Smem {
  uint64_t full[4];
  uint64_t empty[4];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int zero;
};

__device__ __forceinline__ void decode_tile(int t, const int* ts, const int32_t* off_al, int E,
                                            int& e, int& m, int& n) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ts[mid] <= t) lo = mid; else hi = mid - 1;
  }
  e = lo;
  const int mt = (off_al[e + 1] - off_al[e]) / kTileM;
  const int local = t - ts[e];
  n = local / mt;
  m = local - n * mt;
}

template <bool kSwiglu>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1, GroupedGemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  Smem* sm = reinterpret_cast<Smem*>(ring + S * kStageBytes);
  int* ts = reinterpret_cast<int*>(sm + 1);  // [E+1] first tile of each expert
  const int warp = threadIdx.x >> 5, lane = lane_id();
  const int E = p.E;
  const int n_tiles = p.N / p.bn;
  const int kblocks = p.K / BK;
  const int bn = kSwiglu ? 256 : p.bn;       // MMA N (fc1: gate 128 + up 128)
  const uint32_t stage_tx = kABytes + (bn / 64) * kBBox;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm->tfull[a]), 1);
      mbar_init(smem_u32(&sm->tempty[a]), 4 * 32);
    }
    mbar_init(smem_u32(&sm->drain), 1);
    sm->abort = 0;
    sm->zero = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    if (kSwiglu) tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  for (int e = threadIdx.x; e < E; e += kThreads)
    ts[e + 1] = (p.off_al[e + 1] - p.off_al[e]) / kTileM * n_tiles;
  __syncthreads();
  if (threadIdx.x == 0) {
    ts[0] = 0;
    for (int e = 0; e < E; ++e) ts[e + 1] += ts[e];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_base;
  const int total = ts[E];
  volatile int* abort_flag = &sm->abort;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t last_par[4] = {0, 0, 0, 0};
      bool used[4] = {false, false, false, false};
      bool ok = true;
      // the routed rows are re-read by every N tile of their expert: keep them in L2
      const uint64_t pol_a = l2_policy_evict_last();
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int e, m, n;
        decode_tile(t, ts, p.off_al, E, e, m, n);
        const int a_row = p.off_al[e] + m * kTileM;
        const int b_row = e * p.K;
        const int n0 = n * p.bn;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t full = smem_u32(&sm->full[stage]);
          if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full, stage_tx);
          uint8_t* sa = ring + stage * kStageBytes;
          uint8_t* sb = sa + kABytes;
          tma_load_2d_hint(smem_u32(sa), &tmA, full, kb * BK, a_row, pol_a);
          if (kSwiglu) {
            tma_load_2d(smem_u32(sb), &tmB0, full, n0, b_row + kb * BK);
            tma_load_2d(smem_u32(sb + kBBox), &tmB0, full, n0 + 64, b_row + kb * BK);
            tma_load_2d(smem_u32(sb + 2 * kBBox), &tmB1, full, n0, b_row + kb * BK);
            tma_load_2d(smem_u32(sb + 3 * kBBox), &tmB1, full, n0 + 64, b_row + kb * BK);
          } else {
            for (int j = 0; j < bn / 64; ++j)
              tma_load_2d(smem_u32(sb + j * kBBox), &tmB0, full, n0 + 64 * j, b_row + kb * BK);
          }
          last_par[stage] = phase;
          used[stage] = true;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        sm->abort = 1;
        report_error(p.err, kErrTimeout);
      }
      // every issued copy must land before the CTA may exit
      for (int s = 0; s < S; ++s)
        if (used[s]) mbar_wait(smem_u32(&sm->full[s]), last_par[s], kDrainNs, &sm->zero);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kTileM, bn, false, true);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        if (!mbar_wait(smem_u32(&sm->tempty[acc]), acc_phase ^ 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ring + stage * kStageBytes);
          const uint32_t b0 = a0 + kABytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            // A: K-major, 128B swizzle, 8-row groups 1024 B apart; +32 B per K=16.
            const uint64_t ad = sdesc_sw128(a0 + ks * 32, 16, 1024);
            // B: N-major, 128B swizzle; 64-column atoms 8 KB apart (LBO),
            // 8-row K groups 1024 B apart (SBO); +16 rows = 2 KB per K=16.
            const uint64_t bd = sdesc_sw128(b0 + ks * 2048, kBBox, 1024);
            umma_bf16(d, ad, bd, idesc, (kb | ks) ? 1u : 0u);
          }
          umma_commit(smem_u32(&sm->empty[stage]));
          issued = true;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&sm->tfull[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) {
        sm->abort = 1;
        report_error(p.err, kErrTimeout);
      }
      if (issued) {
        umma_commit(smem_u32(&sm->drain));
        mbar_wait(smem_u32(&sm->drain), 0, kDrainNs, &sm->zero);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;                   // TMEM lane quadrant of this warp
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int e, m, n;
      decode_tile(t, ts, p.off_al, E, e, m, n);
      const int64_t grow = p.off_al[e] + m * kTileM + row_in_tile;
      const bool got = mbar_wait(smem_u32(&sm->tfull[acc]), acc_phase, p.wait_ns, abort_flag);
      // tcgen05.ld is warp-collective: the whole warp goes on or stops together
      if (!__all_sync(0xffffffffu, got)) {
        sm->abort = 1;
        if (lane == 0) report_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256;
      if (kSwiglu) {
        __nv_bfloat16* out = p.out + grow * p.N + n * p.bn;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(taddr + c, g);
          tmem_ld_32x32b_x32(taddr + 128 + c, u);
          tmem_ld_wait();
          uint32_t hw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            hw[i] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_global_v4(out + c + 8 * i, hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
          if (p.save_g) {
            __nv_bfloat16* og = p.save_g + grow * p.N + n * p.bn + c;
            __nv_bfloat16* ou = p.save_u + grow * p.N + n * p.bn + c;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              st_global_v4(og + 8 * i,
                           pack_bf16x2(__uint_as_float(g[8 * i]), __uint_as_float(g[8 * i + 1])),
                           pack_bf16x2(__uint_as_float(g[8 * i + 2]), __uint_as_float(g[8 * i + 3])),
                           pack_bf16x2(__uint_as_float(g[8 * i + 4]), __uint_as_float(g[8 * i + 5])),
                           pack_bf16x2(__uint_as_float(g[8 * i + 6]), __uint_as_float(g[8 * i + 7])));
              st_global_v4(ou + 8 * i,
                           pack_bf16x2(__uint_as_float(u[8 * i]), __uint_as_float(u[8 * i + 1])),
                           pack_bf16x2(__uint_as_float(u[8 * i + 2]), __uint_as_float(u[8 * i + 3])),
                           pack_bf16x2(__uint_as_float(u[8 * i + 4]), __uint_as_float(u[8 * i + 5])),
                           pack_bf16x2(__uint_as_float(u[8 * i + 6]), __uint_as_float(u[8 * i + 7])));
            }
          }
        }
      } else {
        __nv_bfloat16* out = p.out + grow * p.N + n * p.bn;
#pragma unroll 1
        for (int c = 0; c < bn; c += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_global_v4(out + c + 8 * i,
                         pack_bf16x2(__uint_as_float(r[8 * i]), __uint_as_float(r[8 * i + 1])),
                         pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                         pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                         pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->tempty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

size_t gemm_smem_bytes(int stages, int E) {
  return 1024 + static_cast<size_t>(stages) * kStageBytes + sizeof(Smem) +
         static_cast<size_t>(E + 1) * sizeof(int);
}

template <bool kSwiglu>
cudaError_t launch_impl(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  // always the 4-stage size: one CTA per SM, so the 512-column TMEM
  // allocation never waits on a neighbour
  const size_t smem = gemm_smem_bytes(4, p.E);
  static size_t configured = 0;
  if (configured < smem) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kSwiglu>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(gemm_smem_bytes(4, kMaxExperts)));
    if (e != cudaSuccess) return e;
    configured = gemm_smem_bytes(4, kMaxExperts);
  }
  grouped_gemm_kernel<kSwiglu><<<grid, kThreads, smem, st>>>(a, b0, b1, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fc1_swiglu(const CUtensorMap& a, const CUtensorMap& wg, const CUtensorMap& wu,
                              const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  return launch_impl<true>(a, wg, wu, p, grid, st);
}

cudaError_t launch_fc2(const CUtensorMap& a, const CUtensorMap& w, const GroupedGemmArgs& p,
                       int grid, cudaStream_t st) {
  return launch_impl<false>(a, w, w, p, grid, st);
}

}  // namespace moe
