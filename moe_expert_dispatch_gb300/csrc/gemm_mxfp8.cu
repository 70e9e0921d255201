// gemm_mxfp8.cu - persistent grouped GEMMs of the MXFP8 expert block on the
// block-scaled tensor cores of sm_103a (tcgen05.mma.kind::mxf8f6f4 with one
// E8M0 scale per 32 elements of K on both operands).
//
// The structure is the one of gemm_bf16.cu (TMA producer warp, single-thread
// MMA issuer, double-buffered TMEM accumulators, four epilogue warps, a ring
// of `stages` shared-memory slots), with these differences:
//   * a k-block is 128 E4M3 elements (128 bytes, one 128B-swizzle row);
//     A (128 rows) and B (128 rows) are both K-major;
//   * the scales of a k-block, one 512-byte atom for A and one for B, arrive
//     by 1D bulk copies into the same slot and are moved into tensor memory
//     with tcgen05.cp (32x128b, replicated over the four lane quadrants);
//     each of the four MMAs of the k-block (K = 32) picks its byte of the
//     32-bit scale words through the instruction's scale-factor id;
//   * accumulators are 128 columns wide (2 x 128), and 8 columns per slot
//     hold that slot's scales, all inside one 512-column allocation;
//   * slots are smaller (34 KB), so the ring is up to 6 deep: at the FP8 rate
//     4 slots in flight per SM do not cover the L2 latency;
//   * fc1's epilogue rounds h to bf16 and quantises it per 32 along F (codes
//     + tiled scales for fc2); fc2's epilogue rounds O to bf16.
// Tiles follow the Rows schedule of gemm_bf16.cu: expert segments padded to
// 128 rows, M fastest within an expert unless it has more M tiles than N
// tiles, CTA b takes tiles b, b + grid, ...
#include "common.cuh"
#include "internal.h"
#include "mx.cuh"

namespace moe {

namespace {

constexpr int BK = 128;                    // E4M3 elements (bytes) per k-block
constexpr int kABytes = kTileM * BK;       // 16 KB
constexpr int kSfBytes = 512;              // one scale atom (128 rows x 4 blocks of 32)
// warp 0 producer, warp 1 MMA issuer, then the epilogue warps. fc1's
// epilogue (SwiGLU + quantisation) is heavy: 8 warps, two per TMEM lane
// quadrant, each finishing half of the tile's columns, halve its exposed
// part. fc2's (bf16 stores) is light: 4 warps (more only take issue slots
// from the producer and MMA threads).
template <bool kFc1>
constexpr int epi_warps() { return kFc1 ? 8 : 4; }
template <bool kFc1>
constexpr int num_threads() { return 64 + 32 * epi_warps<kFc1>(); }
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kDrainNs = 1000000000ull;

constexpr int kMaxStages = 6;

// Tile geometry for an MMA N of 128 or 256. N=128: two accumulators of 128
// columns (the epilogue of a tile overlaps the next tile) and 34 KB slots;
// N=256: one accumulator of 256 columns (no overlap, but half the A reads
// per FLOP) and 50 KB slots. Scales take 4 + N/32 columns per slot after the
// accumulators.
template <int kN>
struct MxGeo {
  static constexpr int kBBytes = kN * BK;
  static constexpr int kSfbAtoms = kN / 128;
  static constexpr int kStageBytes = ((kABytes + kBBytes + (1 + kSfbAtoms) * kSfBytes) + 1023) /
                                     1024 * 1024;
  static constexpr int kAccBufs = kN == 128 ? 2 : 1;
  static constexpr uint32_t kSfCol = kAccBufs * kN;
  static constexpr uint32_t kSfColsPerStage = 4 + 4 * kSfbAtoms;
  static constexpr int kStages = kN == 128 ? 6 : 4;   // what fits in shared memory
};

struct Smem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int zero;
};

template <bool kFc1, int kTileN>
__global__ void __launch_bounds__(num_threads<kFc1>(), 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, MxGemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using G = MxGeo<kTileN>;
  constexpr int kBBytes = G::kBBytes;
  constexpr int kStageBytes = G::kStageBytes;
  const int S = p.stages < G::kStages ? p.stages : G::kStages;
  Smem* sm = reinterpret_cast<Smem*>(ring + S * kStageBytes);
  int* ts = reinterpret_cast<int*>(sm + 1);
  const int warp = threadIdx.x >> 5, lane = lane_id();
  const int E = p.E;
  const int n_cols = kFc1 ? kTileN / 2 : kTileN;   // output columns per N tile
  const int n_tiles = p.N / n_cols;
  const int kblocks = p.K / BK;
  const int kgroups = p.K >> 7;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm->tfull[a]), 1);
      mbar_init(smem_u32(&sm->tempty[a]), epi_warps<kFc1>() * 32);
    }
    mbar_init(smem_u32(&sm->drain), 1);
    sm->abort = 0;
    sm->zero = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  for (int e = threadIdx.x; e < E; e += num_threads<kFc1>())
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

  auto decode = [&](int t, int& e, int& m, int& n) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ts[mid] <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int mt = (p.off_al[e + 1] - p.off_al[e]) / kTileM;
    const int local = t - ts[e];
    if (mt > n_tiles) {       // tall expert: keep its row panel in L2
      m = local / n_tiles;
      n = local - m * n_tiles;
    } else {
      n = local / mt;
      m = local - n * mt;
    }
  };

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t fills = 0;
      bool ok = true;
      const uint64_t pol_a = p.keep_a ? l2_policy_evict_last() : l2_policy_evict_normal();
      const uint32_t ring0 = smem_u32(ring);
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int e, m, n;
        decode(t, e, m, n);
        const int row0 = p.off_al[e] + m * kTileM;
        const int64_t vrow = static_cast<int64_t>(e) * p.sfb_rows + static_cast<int64_t>(n) * kTileN;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t full = smem_u32(&sm->full[stage]);
          if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full, kABytes + kBBytes + (1 + G::kSfbAtoms) * kSfBytes);
          const uint32_t sa = ring0 + stage * kStageBytes;
          const uint32_t sb = sa + kABytes;
          const uint32_t ssf = sb + kBBytes;
          tma_load_2d_hint(sa, &tmA, full, kb * BK, row0, pol_a);
          if (kFc1) {       // N/2 gate rows, then N/2 up rows, of the same N tile
            const int half = kTileN / 2;
            tma_load_2d(sb, &tmB0, full, kb * BK, e * p.b_rows + n * half);
            tma_load_2d(sb + half * BK, &tmB1, full, kb * BK, e * p.b_rows + n * half);
          } else {
            for (int j = 0; j < kTileN; j += 128)
              tma_load_2d(sb + j * BK, &tmB0, full, kb * BK, e * p.b_rows + n * kTileN + j);
          }
          bulk_copy_g2s(ssf, p.sfa + ((static_cast<int64_t>(row0) >> 7) * kgroups + kb) * kSfBytes,
                        kSfBytes, full);
#pragma unroll
          for (int j = 0; j < G::kSfbAtoms; ++j)
            bulk_copy_g2s(ssf + (1 + j) * kSfBytes,
                          p.sfb + (((vrow >> 7) + j) * kgroups + kb) * kSfBytes, kSfBytes, full);
          ++fills;
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
      // the last S fills must land before exit (fill i: slot i % S, parity (i / S) & 1)
      for (uint32_t i = fills > static_cast<uint32_t>(S) ? fills - S : 0; i < fills; ++i)
        mbar_wait(smem_u32(&sm->full[i % S]), (i / S) & 1, kDrainNs, &sm->zero);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
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
        const uint32_t d = tmem_base + acc * kTileN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring) + stage * kStageBytes;
          const uint32_t sb = sa + kABytes;
          const uint32_t ssf = sb + kBBytes;
          // this slot's scales into its own TMEM columns: A at +0..3, B's
          // 128-row atoms at +4..7 (and +8..11 for N = 256)
          const uint32_t sfa_t = tmem_base + G::kSfCol + stage * G::kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + 4;
          tmem_cp_32x128b_warpx4(sfa_t, sdesc_noswizzle(ssf, 16, 128));
#pragma unroll
          for (int j = 0; j < G::kSfbAtoms; ++j)
            tmem_cp_32x128b_warpx4(sfb_t + 4 * j,
                                   sdesc_noswizzle(ssf + (1 + j) * kSfBytes, 16, 128));
          const uint64_t ad = sdesc_sw128(sa, 16, 1024), bd = sdesc_sw128(sb, 16, 1024);
#pragma unroll
          for (int ks = 0; ks < BK / 32; ++ks)      // +32 B of K per MMA
            umma_mxf8(d, ad + 2 * ks, bd + 2 * ks, idesc_mxf8(kTileM, kTileN, ks, ks), sfa_t,
                      sfb_t, (kb | ks) ? 1u : 0u);
          umma_commit(smem_u32(&sm->empty[stage]));
          issued = true;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&sm->tfull[acc]));
        if (++acc == G::kAccBufs) {
          acc = 0;
          acc_phase ^= 1;
        }
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
    const int half = (warp - 2) >> 2;         // fc1: which half of the tile's columns
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int e, m, n;
      decode(t, e, m, n);
      const int64_t grow = p.off_al[e] + m * kTileM + row_in_tile;
      const bool got = mbar_wait(smem_u32(&sm->tfull[acc]), acc_phase, p.wait_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        sm->abort = 1;
        if (lane == 0) report_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kTileN;
      // The whole accumulator row is read into registers (packed bf16, or
      // the finished E4M3 codes for fc1) and the accumulator is released
      // before any global store, so that with a single accumulator the
      // stores still overlap the next tile's MMAs.
      if (kFc1) {
        // h = bf16(silu(gate) * up), then MXFP8 per 32 along F. The tile's
        // N/64 scale bytes of this row are adjacent in the tiled layout (one
        // 128-wide K group of fc2): they leave in one store.
        // this warp's half of the tile's h columns: kTileN / 4 of them
        constexpr int kHalf = kTileN / 4;
        const int c0 = half * kHalf;
        uint32_t codes[kHalf / 4];
        uint32_t packed = 0;
#pragma unroll
        for (int c = 0; c < kHalf; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(taddr + c0 + c, g);
          tmem_ld_32x32b_x32(taddr + kTileN / 2 + c0 + c, u);
          tmem_ld_wait();
          float hv[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            hv[i] = __bfloat162float(__float2bfloat16_rn(silu_f(__uint_as_float(g[i])) *
                                                         __uint_as_float(u[i])));
          const uint8_t sc = quantize_block32(hv, &codes[c / 4]);
          packed |= static_cast<uint32_t>(sc) << (8 * (c >> 5));
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&sm->tempty[acc]));
        const int col = n * n_cols + c0;
        int4* dst = reinterpret_cast<int4*>(p.hq + grow * p.N + col);
#pragma unroll
        for (int i = 0; i < kHalf / 16; ++i)
          dst[i] = make_int4(codes[4 * i], codes[4 * i + 1], codes[4 * i + 2], codes[4 * i + 3]);
        uint8_t* hs = p.hs + mx_scale_offset(grow, col >> 5, p.N);
        if (kHalf == 64)
          *reinterpret_cast<uint16_t*>(hs) = static_cast<uint16_t>(packed);
        else
          *hs = static_cast<uint8_t>(packed);
      } else {
        constexpr int kHalf = kTileN;           // this warp's columns: all of them
        const int c0 = 0;
        uint32_t w[kHalf / 2];
#pragma unroll
        for (int c = 0; c < kHalf; c += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c0 + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[c / 2 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&sm->tempty[acc]));
        __nv_bfloat16* out = p.out + grow * p.N + n * kTileN + c0;
#pragma unroll
        for (int i = 0; i < kHalf / 8; ++i)
          st_global_v4(out + 8 * i, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
      if (++acc == G::kAccBufs) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool kFc1, int kN>
cudaError_t launch_mx(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                      const MxGemmArgs& p, int grid, cudaStream_t st) {
  using G = MxGeo<kN>;
  const size_t smem = 1024 + G::kStages * static_cast<size_t>(G::kStageBytes) + sizeof(Smem) +
                      static_cast<size_t>(kMaxExperts + 1) * sizeof(int);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel<kFc1, kN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  mx_gemm_kernel<kFc1, kN><<<grid, num_threads<kFc1>(), smem, st>>>(a, b0, b1, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mx_fc1(const CUtensorMap& a, const CUtensorMap& wg, const CUtensorMap& wu,
                          const MxGemmArgs& p, int grid, cudaStream_t st) {
  return p.bn == 256 ? launch_mx<true, 256>(a, wg, wu, p, grid, st)
                     : launch_mx<true, 128>(a, wg, wu, p, grid, st);
}

cudaError_t launch_mx_fc2(const CUtensorMap& a, const CUtensorMap& wd, const MxGemmArgs& p,
                          int grid, cudaStream_t st) {
  return p.bn == 256 ? launch_mx<false, 256>(a, wd, wd, p, grid, st)
                     : launch_mx<false, 128>(a, wd, wd, p, grid, st);
}

}  // namespace moe
