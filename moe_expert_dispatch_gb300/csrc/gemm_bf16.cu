// gemm_bf16.cu - persistent grouped GEMMs of the expert block on the
// 5th-generation tensor cores (tcgen05) of sm_103a, forward and backward.
//
// Structure (one CTA per SM, 6 warps):
//   warp 0      TMA producer: streams the A tile (128 x 64 of K) and the B
//               tile (64 of K x bn) of every k-block into a ring of
//               `stages` shared-memory slots of 48 KB.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=bn,
//               K=16) on each slot and releases it with tcgen05.commit; it
//               accumulates a tile in one of two TMEM buffers (2 x 256
//               columns) so that the epilogue of tile i overlaps tile i+1.
//   warps 2-5   epilogue: tcgen05.ld the accumulator and finish the tile.
// This is the in-kernel counterpart of the MC2 ring of "MC2 通算融合架构总览"
// (sections 3-4): the producer's TMA loads stand where the AIV's UDMA puts
// stood, the full/empty mbarrier pair where the CrossCore set/wait flags
// stood, and slot = k-block mod stages as bufferId = mLoopIdx mod bufferSize.
//
// CTA pairs (kPair, Rows schedules): the two CTAs of a cluster of two share
// one tile of M = 256 (tcgen05.mma.cta_group::2). Each CTA loads its own 128
// rows of A and half of the tile's B columns (gate or up of fc1, one half of
// the N tile otherwise) into its own ring, so each SM streams half the B
// bytes of a one-CTA tile for the same FLOPs; the slots (32 KB) are smaller,
// and the ring is 6 deep. Both CTAs' copies complete on the leader's (rank
// 0) full barrier, the leader's thread issues the MMAs, and their commits
// release the slots and hand the accumulators to the epilogues of both CTAs;
// each CTA finishes its own 128 rows. An expert whose segment has an odd
// number of 128-row blocks ends in a tile whose second half lies past the
// expert: there the second CTA loads no A rows and stores nothing.
//
// Two schedules share the kernel:
//  * Rows (fc1, fc2, dH, dXp): expert e owns rows [off_al[e], off_al[e+1])
//    of the permuted activations, a multiple of 128 (padded), i.e. one M
//    tile per 128 rows, times N/bn N tiles; the reduction is a fixed K.
//  * WGrad (dW1, dW2): expert e owns (M/128) x (N/bn) tiles of its weight
//    gradient and the reduction runs over its (zero-padded) rows.
// Tiles of all experts are numbered consecutively and CTA b takes tiles b,
// b + grid, ...; within an expert the dimension of the larger operand runs
// fastest, so that the smaller operand's panels are the ones re-read from
// L2: in Rows, M fastest (CTAs that run at the same time share one weight
// tile) unless the expert has more M tiles than N tiles; in WGrad, N fastest
// when M > N (dW2: the h panels stream once) and M fastest otherwise (dW1).
// Experts without rows own no Rows tile. Counts never leave the device.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int BK = 64;                         // k-block (128 bytes of bf16)
constexpr int kABytes = kTileM * BK * 2;       // 16 KB
constexpr int kBBox = 64 * BK * 2;             // 8 KB: 64 columns x 64 of K
// A slot holds A and the CTA's B columns of the widest tile (N = 256): all of
// them for one CTA (48 KB, 4 slots), half of them for a CTA of a pair (32 KB,
// 6 slots).
template <bool kPair>
constexpr int stage_bytes() { return kABytes + (kPair ? 2 : 4) * kBBox; }
template <bool kPair>
constexpr int max_stages() { return kPair ? 6 : 4; }
constexpr int kThreads = 192;
// fc1 with the fused gather: warp 0 and the added warps 6.. gather, each
// copying 128 / kGatherWarps of the tile's token rows
constexpr int kGatherWarps = 2;
template <bool kGather>
constexpr int block_threads() { return kGather ? kThreads + 32 * (kGatherWarps - 1) : kThreads; }
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kDrainNs = 1000000000ull;
constexpr unsigned long long kPairDrainNs = 50000000ull;

struct Smem {
  uint64_t full[6];
  uint64_t empty[6];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int zero;
};

struct Tile {
  int e, m, n;
  int row0;      // Rows: first A row (of the pair's tile); WGrad: first reduction row
  int kblocks;
  int half_rows; // pairs: 128-row blocks of the tile inside the expert (1 or 2)
};

// M tiles of an expert with mt 128-row blocks: one per block, or one per two
// blocks for CTA pairs (the last one half-filled when mt is odd).
template <bool kPair>
__device__ __forceinline__ int m_tiles(int mt) { return kPair ? (mt + 1) >> 1 : mt; }

template <Sched kSched, bool kPair>
__device__ __forceinline__ Tile decode_tile(int t, const int* ts, const GroupedGemmArgs& p) {
  Tile tl;
  tl.half_rows = 1;
  if (kSched == Sched::Rows) {
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ts[mid] <= t) lo = mid; else hi = mid - 1;
    }
    tl.e = lo;
    const int mb = (p.off_al[tl.e + 1] - p.off_al[tl.e]) / kTileM;
    const int mt = m_tiles<kPair>(mb);
    const int nt = p.N / (p.b_split == 1 ? p.bn / 2 : p.bn);
    const int local = t - ts[tl.e];
    if (mt > nt) {            // tall expert: its row panel is the larger operand, keep it in L2
      tl.m = local / nt;
      tl.n = local - tl.m * nt;
    } else {                  // the weight panel is larger: M fastest shares it between CTAs
      tl.n = local / mt;
      tl.m = local - tl.n * mt;
    }
    tl.row0 = p.off_al[tl.e] + tl.m * (kPair ? 2 * kTileM : kTileM);
    if (kPair) tl.half_rows = min(2, mb - 2 * tl.m);
    tl.kblocks = p.K / BK;
  } else {
    const int mt = p.M / (kPair ? 2 * kTileM : kTileM);   // pairs: M % 256 == 0
    const int nt = p.N / p.bn;
    const int per = mt * nt;
    tl.e = t / per;
    const int local = t - tl.e * per;
    if (p.M > p.N) {          // A (M x K) is the larger operand: N fastest keeps B's panels in L2
      tl.m = local / nt;
      tl.n = local - tl.m * nt;
    } else {                  // B is larger: M fastest keeps A's panels in L2
      tl.n = local / mt;
      tl.m = local - tl.n * mt;
    }
    tl.row0 = p.off_al[tl.e];
    tl.kblocks = (p.off_al[tl.e + 1] - tl.row0) / BK;
    if (kPair) tl.half_rows = 2;   // M % 256 == 0: both halves lie inside the gradient
  }
  return tl;
}

// Epilogue output pieces: each epilogue warp finishes its 32 rows of the
// tile in pieces of 32 rows x 64 bytes (32 bf16 or 16 float columns), staged
// in its own shared-memory slots with the 64-byte swizzle (16-byte chunk j
// of row r at chunk j ^ ((r >> 1) & 3): a warp's row writes take 4
// wavefronts, the minimum for 512 bytes) and stored by its lane 0 with a TMA
// tensor store. Warps never wait for each other.
constexpr int kPieceBytes = 32 * 64;       // 2 KB
constexpr int kSlotsPerWarp = 3;
constexpr int kPieceArea = 4 * kSlotsPerWarp * kPieceBytes;   // 24 KB

template <Epi kEpi, bool kAmn, bool kBmn, Sched kSched, bool kGather, int kBN, bool kPair>
__global__ void __launch_bounds__(block_threads<kGather>(), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmO0,
                        const __grid_constant__ CUtensorMap tmO1,
                        const __grid_constant__ CUtensorMap tmO2, GroupedGemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  static_assert(!kPair || (!kGather && (kSched == Sched::Rows ? !kAmn : (kAmn && kBmn))),
                "CTA pairs: the Rows schedule with a K-major A, or WGrad");
  constexpr int kStageBytes = stage_bytes<kPair>();
  const int S = p.stages;
  uint8_t* pieces = ring + max_stages<kPair>() * kStageBytes;  // after the largest ring
  Smem* sm = reinterpret_cast<Smem*>(pieces + kPieceArea);
  int* ts = reinterpret_cast<int*>(sm + 1);  // [E+1] first tile of each expert (Rows)
  const int warp = threadIdx.x >> 5, lane = lane_id();
  const int E = p.E;
  constexpr int bn = kBN;                     // MMA N
  const int n_tiles = p.N / (kEpi == Epi::SwigluFwd ? bn / 2 : bn);
  constexpr uint32_t stage_tx = kABytes + (bn / 64) * kBBox;   // one-CTA tile
  // CTA pairs: this CTA's rank, the tile walk over clusters, and the
  // leader's barriers as seen from either CTA
  const uint32_t rank = kPair ? cluster_ctarank() : 0;
  const int walk0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int walk_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // gathering: the producer's expect_tx arrival and one cp.async
      // arrival per lane of the gathering warps
      mbar_init(smem_u32(&sm->full[s]), kGather ? 1 + 32 * kGatherWarps : 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm->tfull[a]), 1);
      // one arrival per epilogue warp (of both CTAs of a pair: the leader's
      // MMAs overwrite both CTAs' accumulators)
      mbar_init(smem_u32(&sm->tempty[a]), kPair ? 8 : 4);
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
    tma_prefetch_desc(&tmO0);
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(smem_u32(&sm->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  int total;
  if (kSched == Sched::Rows) {
    for (int e = threadIdx.x; e < E; e += block_threads<kGather>())
      ts[e + 1] = m_tiles<kPair>((p.off_al[e + 1] - p.off_al[e]) / kTileM) * n_tiles;
    __syncthreads();
    if (threadIdx.x == 0) {
      ts[0] = 0;
      for (int e = 0; e < E; ++e) ts[e + 1] += ts[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();   // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_base;
  if (kSched == Sched::Rows) total = ts[E];
  else total = E * (p.M / (kPair ? 2 * kTileM : kTileM)) * n_tiles;
  volatile int* abort_flag = &sm->abort;

  if (kGather && (warp == 0 || warp >= 6)) {
    // ---------------------------------------------------------- gathering producer
    // kGatherWarps warps gather the A tile's 128 token rows of x (64 columns,
    // 128 bytes each) with cp.async, an equal share each: per warp instruction
    // 4 rows of 8 lanes x 16 bytes (lane l of gathering warp g: row
    // g * 128 / kGatherWarps + 4i + l / 8, chunk l % 8), written
    // swizzled as a tiled 128B-swizzle load would (chunk c of row r at
    // c ^ (r & 7)); each lane then arrives on the slot's barrier once its
    // copies have landed. Lane 0 of warp 0 also loads the weight boxes by TMA. This is the dispatch AllToAllv of
    // all2all_grouped_matmul folded into the GEMM's producer. (TMA gather4,
    // four rows per instruction, was bound by the TMA unit's rate at 3.4x the
    // materialised permute.)
    int stage = 0;
    uint32_t phase = 0;
    uint32_t fills = 0;
    bool ok = true;
    const int chunk = lane & 7;
    const int g0 = (warp == 0 ? 0 : warp - 5) * (128 / kGatherWarps);   // first row of the tile
    constexpr int kRows = 128 / kGatherWarps / 4;   // rows per lane
    const bool lead = warp == 0 && lane == 0;
    for (int t = walk0; t < total && ok; t += walk_step) {
      const Tile tl = decode_tile<kSched, kPair>(t, ts, p);
      const int real_end = p.off_al[tl.e] + p.counts[tl.e];
      const __nv_bfloat16* src[kRows];          // this lane's rows, at column 0
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const int r = tl.row0 + g0 + 4 * i + (lane >> 3);
        const int tok = r < real_end ? __ldg(p.gather_token + r) : 0;   // padding: any valid row
        src[i] = p.gather_x + static_cast<int64_t>(tok) * p.K + chunk * 8;
      }
      const int krow = tl.e * static_cast<int>(p.b_rows);
      const int n0 = tl.n * (bn / 2);
      for (int kb = 0; kb < tl.kblocks; ++kb) {
        const uint32_t full = smem_u32(&sm->full[stage]);
        const bool got = mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.wait_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(ring + stage * kStageBytes);
        const uint32_t sb = sa + kABytes;
        if (lead) {
          mbar_arrive_expect_tx(full, (bn / 64) * kBBox);
          for (int j = 0; j < bn / 128; ++j) {
            tma_load_2d(sb + j * kBBox, &tmB0, full, n0 + 64 * j, krow + kb * BK);
            tma_load_2d(sb + (bn / 128 + j) * kBBox, &tmB1, full, n0 + 64 * j, krow + kb * BK);
          }
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          const int r = g0 + 4 * i + (lane >> 3);
          cp_async_16(sa + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * BK);
        }
        cp_async_arrive_noinc(full);
        ++fills;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      sm->abort = 1;
      report_error(p.err, kErrTimeout);
    }
    // every issued copy must land before the CTA may exit: the last S fills
    // (fill i went to slot i % S with phase parity (i / S) & 1)
    if (lane == 0)
      for (uint32_t i = fills > static_cast<uint32_t>(S) ? fills - S : 0; i < fills; ++i)
        mbar_wait(smem_u32(&sm->full[i % S]), (i / S) & 1, kDrainNs, &sm->zero);
  } else if (warp == 0) {
    // ---------------------------------------------------------- producer
    // One thread; it is on the critical path of every k-block, so the loop
    // body is straight-line: box counts are compile-time, the L2 policy of A
    // is a value chosen once (operands re-read by many tiles of their expert
    // stay in L2 longer when all of A fits there; pinning a larger operand
    // would push the weights out instead).
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t fills = 0;
      bool ok = true;
      const uint64_t pol_a = p.keep_a ? l2_policy_evict_last() : l2_policy_evict_normal();
      const uint64_t pol_b = l2_policy_evict_normal();
      const uint32_t ring0 = smem_u32(ring);
      for (int t = walk0; t < total && ok; t += walk_step) {
        const Tile tl = decode_tile<kSched, kPair>(t, ts, p);
        // per-tile coordinates; a CTA of a pair takes the second 128 rows of
        // the pair's M tile when its rank is 1 (Rows: rows of A; WGrad: the
        // columns of the MN-major A)
        const int m128 = kPair ? 2 * tl.m + static_cast<int>(rank) : tl.m;
        const int a_x0 = kAmn ? m128 * kTileM : 0;
        const int a_y0 = (kPair && !kAmn) ? tl.row0 + static_cast<int>(rank) * kTileM : tl.row0;
        const int b_row0 = (kSched == Sched::Rows) ? tl.e * static_cast<int>(p.b_rows) : tl.row0;
        const int b_n0 = (kEpi == Epi::SwigluFwd) ? tl.n * (bn / 2) : tl.n * bn;
        // pairs: the second CTA's rows may lie past the expert (odd tail)
        const bool load_a = !kPair || static_cast<int>(rank) < tl.half_rows;
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          const uint32_t full = smem_u32(&sm->full[stage]);
          if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t sa = ring0 + stage * kStageBytes;
          const uint32_t sb = sa + kABytes;
          const int k0 = kb * BK;
          if constexpr (kPair) {
            // both CTAs' copies complete on the leader's full barrier, which
            // the leader arms with the bytes of the whole pair tile
            const uint32_t full_l = mapa_shared(full, 0);
            if (rank == 0)
              mbar_arrive_expect_tx(full, tl.half_rows * kABytes + (bn / 64) * kBBox);
            if (load_a) {
              if (kAmn) {     // MN-major A: two boxes of 64 of M x 64 of K
                tma_load_2d_pair(sa, &tmA, full_l, a_x0, a_y0 + k0, pol_a);
                tma_load_2d_pair(sa + kBBox, &tmA, full_l, a_x0 + 64, a_y0 + k0, pol_a);
              } else {
                tma_load_2d_pair(sa, &tmA, full_l, k0, a_y0, pol_a);
              }
            }
            if (kBmn) {       // this CTA's half of the N tile: bn / 128 boxes of 64 columns
              const int krow = b_row0 + k0;
              const CUtensorMap* mb = (kEpi == Epi::SwigluFwd && rank == 1) ? &tmB1 : &tmB0;
              const int n0 = (kEpi == Epi::SwigluFwd) ? b_n0 : b_n0 + static_cast<int>(rank) * (bn / 2);
#pragma unroll
              for (int j = 0; j < bn / 128; ++j)
                tma_load_2d_pair(sb + j * kBBox, mb, full_l, n0 + 64 * j, krow, pol_b);
            } else {          // K-major B: this CTA's bn / 2 rows in one box
              const int nrow = b_row0 + b_n0 + static_cast<int>(rank) * (bn / 2);
              if (p.b_split == 2 && kb >= p.k_split)
                tma_load_2d_pair(sb, &tmB1, full_l, k0 - p.k_split * BK, nrow, pol_b);
              else
                tma_load_2d_pair(sb, &tmB0, full_l, k0, nrow, pol_b);
            }
            ++fills;
            if (++stage == S) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          mbar_arrive_expect_tx(full, stage_tx);
          if (!kAmn) {
            tma_load_2d_hint(sa, &tmA, full, k0, a_y0, pol_a);
          } else {
            tma_load_2d_hint(sa, &tmA, full, a_x0, a_y0 + k0, pol_a);
            tma_load_2d_hint(sa + kBBox, &tmA, full, a_x0 + 64, a_y0 + k0, pol_a);
          }
          if (kBmn) {
            const int krow = b_row0 + k0;
            if (kEpi == Epi::SwigluFwd) {    // gate | up halves of one N tile
#pragma unroll
              for (int j = 0; j < bn / 128; ++j) {
                tma_load_2d(sb + j * kBBox, &tmB0, full, b_n0 + 64 * j, krow);
                tma_load_2d(sb + (bn / 128 + j) * kBBox, &tmB1, full, b_n0 + 64 * j, krow);
              }
            } else {
#pragma unroll
              for (int j = 0; j < bn / 64; ++j)
                tma_load_2d(sb + j * kBBox, &tmB0, full, b_n0 + 64 * j, krow);
            }
          } else {                           // K-major B: one box of bn rows
            const int nrow = b_row0 + b_n0;
            if (p.b_split == 2 && kb >= p.k_split)
              tma_load_2d(sb, &tmB1, full, k0 - p.k_split * BK, nrow);
            else
              tma_load_2d(sb, &tmB0, full, k0, nrow);
          }
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
      // every issued copy must land before the CTA may exit: the last S fills
      // (fill i went to slot i % S with phase parity (i / S) & 1). A pair's
      // copies complete on the leader's barrier; here each CTA waits until
      // the MMAs that read its last fills released them (a slot is released
      // only after both CTAs' copies into it landed). After an abort the
      // MMAs may never come, so those waits are short: a copy lands within
      // microseconds.
      for (uint32_t i = fills > static_cast<uint32_t>(S) ? fills - S : 0; i < fills; ++i) {
        if (kPair)
          mbar_wait(smem_u32(&sm->empty[i % S]), (i / S) & 1, kPairDrainNs, &sm->zero);
        else
          mbar_wait(smem_u32(&sm->full[i % S]), (i / S) & 1, kDrainNs, &sm->zero);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {   // pairs: the leader's thread issues for both CTAs
      const uint32_t idesc = idesc_bf16(kPair ? 2 * kTileM : kTileM, bn, kAmn, kBmn);
      // descriptors of slot 0; a slot adds kStageBytes, a K=16 step adds 32 B
      // (K-major) or 16 rows = 2 KB (MN-major) to the 16-byte start field
      const uint32_t ring0 = smem_u32(ring);
      const uint64_t adesc0 = kAmn ? sdesc_sw128(ring0, kBBox, 1024) : sdesc_sw128(ring0, 16, 1024);
      const uint64_t bdesc0 = kBmn ? sdesc_sw128(ring0 + kABytes, kBBox, 1024)
                                   : sdesc_sw128(ring0 + kABytes, 16, 1024);
      constexpr uint64_t kAStep = kAmn ? (2048 >> 4) : (32 >> 4);
      constexpr uint64_t kBStep = kBmn ? (2048 >> 4) : (32 >> 4);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int t = walk0; t < total && ok; t += walk_step) {
        const Tile tl = decode_tile<kSched, kPair>(t, ts, p);
        if (!mbar_wait(smem_u32(&sm->tempty[acc]), acc_phase ^ 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          // a gathered A tile was written through the generic proxy (cp.async):
          // order it before the tensor core's async-proxy reads
          if (kGather) fence_proxy_async_shared();
          tc_fence_after();
          // K-major, 128B swizzle: 8-row groups 1024 B apart, +32 B per K=16.
          // MN-major, 128B swizzle: 64-wide atoms 8 KB apart (LBO), 8-row K
          // groups 1024 B apart (SBO), +16 rows = 2 KB per K=16.
          const uint64_t soff = static_cast<uint64_t>(stage) * (kStageBytes >> 4);
          const uint64_t ad = adesc0 + soff, bd = bdesc0 + soff;
          if constexpr (kPair) {
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              umma_bf16_pair(d, ad + ks * kAStep, bd + ks * kBStep, idesc, (kb | ks) ? 1u : 0u);
            umma_commit_pair_mc(smem_u32(&sm->empty[stage]), 0x3);   // the slot, in both CTAs
          } else {
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              umma_bf16(d, ad + ks * kAStep, bd + ks * kBStep, idesc, (kb | ks) ? 1u : 0u);
            umma_commit(smem_u32(&sm->empty[stage]));
          }
          issued = true;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if (kPair)
          umma_commit_pair_mc(smem_u32(&sm->tfull[acc]), 0x3);   // both CTAs' epilogues
        else
          umma_commit(smem_u32(&sm->tfull[acc]));   // also for a tile with no k-block
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) {
        sm->abort = 1;
        report_error(p.err, kErrTimeout);
      }
      if (issued) {
        if (kPair)
          umma_commit_pair_mc(smem_u32(&sm->drain), 0x1);
        else
          umma_commit(smem_u32(&sm->drain));
        mbar_wait(smem_u32(&sm->drain), 0, kDrainNs, &sm->zero);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;                   // TMEM lane quadrant of this warp
    const uint32_t slot0 = smem_u32(pieces) + q * kSlotsPerWarp * kPieceBytes;
    const uint32_t my_row = lane * 64;
    const uint32_t sw = (lane >> 1) & 3;
    int npiece = 0;
    // a piece: wait for the warp's next slot, fill this lane's row, store it
    auto piece_slot = [&]() -> uint32_t {
      if (lane == 0) bulk_wait_group_read<kSlotsPerWarp - 1>();
      __syncwarp();
      return slot0 + (npiece % kSlotsPerWarp) * kPieceBytes;
    };
    auto put_row = [&](uint32_t slot, const uint32_t* w16) {   // 16 words = 64 bytes
#pragma unroll
      for (int j = 0; j < 4; ++j)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(slot + my_row +
                                                                       ((j ^ sw) << 4)),
                     "r"(w16[4 * j]), "r"(w16[4 * j + 1]), "r"(w16[4 * j + 2]),
                     "r"(w16[4 * j + 3])
                     : "memory");
    };
    auto piece_out = [&](uint32_t slot, const CUtensorMap* map, int x, int y, bool add) {
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        if (add) tma_reduce_add_2d(map, slot, x, y + q * 32);
        else tma_store_2d(map, slot, x, y + q * 32);
        bulk_commit_group();
      }
      ++npiece;
    };
    auto bf16_piece = [&](const uint32_t* f32x32, const CUtensorMap* map, int x, int y) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(__uint_as_float(f32x32[2 * i]), __uint_as_float(f32x32[2 * i + 1]));
      const uint32_t slot = piece_slot();
      put_row(slot, w);
      piece_out(slot, map, x, y, false);
    };
    // a 32 x 32 bf16 block of A_g or A_u in the blocked layout
    // (act_block_offset): lane r's row is its four 16-byte slab pieces, so
    // each warp store writes 512 contiguous bytes straight from registers
    auto put_block = [&](const uint32_t* f32x32, __nv_bfloat16* dst) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(__uint_as_float(f32x32[2 * i]), __uint_as_float(f32x32[2 * i + 1]));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_global_v4(dst + j * 256 + lane * 8, w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    };
    // SwigluBwd: lane r's row of a 32 x 32 block of A_g or A_u, as 16 words
    auto load_act = [&](const __nv_bfloat16* block, uint32_t* w16) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(block + j * 256 + lane * 8));
        w16[4 * j] = static_cast<uint32_t>(v.x);
        w16[4 * j + 1] = static_cast<uint32_t>(v.y);
        w16[4 * j + 2] = static_cast<uint32_t>(v.z);
        w16[4 * j + 3] = static_cast<uint32_t>(v.w);
      }
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    // the accumulator is handed back to the MMA issuer (the leader, for a
    // pair) by one arrival per warp
    const uint32_t tempty0 = kPair ? mapa_shared(smem_u32(&sm->tempty[0]), 0) : 0;
    for (int t = walk0; t < total; t += walk_step) {
      Tile tl = decode_tile<kSched, kPair>(t, ts, p);
      if (kPair && kSched == Sched::Rows)
        tl.row0 += static_cast<int>(rank) * kTileM;   // this CTA's 128 rows
      if (kPair && kSched == Sched::WGrad)
        tl.m = 2 * tl.m + static_cast<int>(rank);     // this CTA's 128 rows of the gradient
      const bool live = !kPair || static_cast<int>(rank) < tl.half_rows;
      // SwigluBwd: the warp's rows of A_g, A_u for the tile's first 32
      // columns arrive while its MMAs run; the other blocks go to L2 now
      uint32_t ag_w[16], au_w[16];
      const int64_t wrow0 = tl.row0 + q * 32;
      if (kEpi == Epi::SwigluBwd && live) {
#pragma unroll 1
        for (int c = 32; c < bn; c += 32)       // 16 lines per block: lanes 0-15 A_g
          prefetch_l2((lane < 16 ? p.act_g : p.act_u) +
                      act_block_offset(wrow0, tl.n * bn + c, p.ld_act) + (lane & 15) * 64);
        load_act(p.act_g + act_block_offset(wrow0, tl.n * bn, p.ld_act), ag_w);
        load_act(p.act_u + act_block_offset(wrow0, tl.n * bn, p.ld_act), au_w);
      }
      const bool got = mbar_wait(smem_u32(&sm->tfull[acc]), acc_phase, p.wait_ns, abort_flag);
      // tcgen05.ld is warp-collective: the whole warp goes on or stops together
      if (!__all_sync(0xffffffffu, got)) {
        sm->abort = 1;
        if (lane == 0) report_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256;
      if (!live) {
        // pairs: rows past the expert; the accumulator holds nothing to keep
      } else if (kEpi == Epi::SwigluFwd) {
        const int n0 = tl.n * (bn / 2);
#pragma unroll 1
        for (int c = 0; c < bn / 2; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(taddr + c, g);
          tmem_ld_32x32b_x32(taddr + bn / 2 + c, u);
          tmem_ld_wait();
          uint32_t hw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            hw[i] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
          }
          const uint32_t slot = piece_slot();
          put_row(slot, hw);
          piece_out(slot, &tmO0, n0 + c, tl.row0, false);
          if (p.save_g) {
            put_block(g, p.save_g + act_block_offset(tl.row0 + q * 32, n0 + c, p.ld_act));
            put_block(u, p.save_u + act_block_offset(tl.row0 + q * 32, n0 + c, p.ld_act));
          }
        }
      } else if (kEpi == Epi::Bf16) {
#pragma unroll 1
        for (int c = 0; c < bn; c += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + c, v);
          tmem_ld_wait();
          bf16_piece(v, &tmO0, tl.n * bn + c, tl.row0);
        }
      } else if (kEpi == Epi::SwigluBwd) {
        // dA_g = bf16(dH A_u s (1 + A_g (1 - s))), dA_u = bf16(dH A_g s), s = sigmoid(A_g);
        // the next 32 columns of A_g, A_u are loaded one step ahead
        const int f0 = tl.n * bn;
#pragma unroll 1
        for (int c = 0; c < bn; c += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + c, v);
          uint32_t ag_n[16], au_n[16];
          if (c + 32 < bn) {
            load_act(p.act_g + act_block_offset(wrow0, f0 + c + 32, p.ld_act), ag_n);
            load_act(p.act_u + act_block_offset(wrow0, f0 + c + 32, p.ld_act), au_n);
          }
          tmem_ld_wait();
          uint32_t wg[16], wu[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float vg[2], vu[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float dh = __uint_as_float(v[2 * i + h]);
              const float a = __uint_as_float(h ? (ag_w[i] & 0xFFFF0000u) : (ag_w[i] << 16));
              const float b = __uint_as_float(h ? (au_w[i] & 0xFFFF0000u) : (au_w[i] << 16));
              const float sg = sigmoid_f(a);
              vg[h] = dh * b * sg * (1.0f + a * (1.0f - sg));
              vu[h] = dh * a * sg;
            }
            wg[i] = pack_bf16x2(vg[0], vg[1]);
            wu[i] = pack_bf16x2(vu[0], vu[1]);
          }
          uint32_t slot = piece_slot();
          put_row(slot, wg);
          piece_out(slot, &tmO0, f0 + c, tl.row0, false);
          slot = piece_slot();
          put_row(slot, wu);
          piece_out(slot, &tmO0, p.out_split + f0 + c, tl.row0, false);
          if (c + 32 < bn) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              ag_w[i] = ag_n[i];
              au_w[i] = au_n[i];
            }
          }
        }
      } else {  // Epi::F32: float rows (Rows) or weight-gradient rows (WGrad)
        const CUtensorMap* map = &tmO0;
        int col = tl.n * bn;
        int y = tl.row0;
        if (kSched == Sched::WGrad) {
          y = tl.e * p.M + tl.m * kTileM;
          if (p.out_split > 0 && col >= p.out_split) {   // second output, same layout
            map = &tmO1;
            col -= p.out_split;
          }
        }
        const bool add = p.accumulate != 0;
        if (tl.kblocks == 0 && add) {
          // an expert without rows adds nothing to the gradients
        } else {
#pragma unroll 1
          for (int c = 0; c < bn; c += 32) {
            uint32_t v[32];
            if (tl.kblocks > 0) {
              tmem_ld_32x32b_x32(taddr + c, v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0u;      // an expert without rows
            }
            uint32_t slot = piece_slot();
            put_row(slot, v);
            piece_out(slot, map, col + c, y, add);
            slot = piece_slot();
            put_row(slot, v + 16);
            piece_out(slot, map, col + c + 16, y, add);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair)
          mbar_arrive_cluster(tempty0 + acc * static_cast<uint32_t>(sizeof(uint64_t)));
        else
          mbar_arrive(smem_u32(&sm->tempty[acc]));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_group_all();     // every store has landed before exit
  }

  tc_fence_before();
  __syncthreads();
  // pairs: neither CTA leaves while the other may still signal its barriers,
  // read its slots (the leader's MMAs) or write its accumulators
  if (kPair) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool kPair>
constexpr size_t gemm_smem_bytes() {
  return 1024 + max_stages<kPair>() * static_cast<size_t>(stage_bytes<kPair>()) + kPieceArea +
         sizeof(Smem) + static_cast<size_t>(kMaxExperts + 1) * sizeof(int);
}
static_assert(gemm_smem_bytes<false>() <= 232448 && gemm_smem_bytes<true>() <= 232448,
              "shared memory of one CTA");

template <Epi kEpi, bool kAmn, bool kBmn, Sched kSched, bool kGather, int kBN, bool kPair>
cudaError_t launch_bn(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                      const GemmOut& o, const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  // always the deepest ring's size: one CTA per SM, so the 512-column TMEM
  // allocation never waits on a neighbour
  const size_t smem = gemm_smem_bytes<kPair>();
  static bool configured[kMaxDevices] = {};    // the attribute is per device
  static int max_pairs[kMaxDevices] = {};      // clusters of two that fit at once
  auto kern = grouped_gemm_kernel<kEpi, kAmn, kBmn, kSched, kGather, kBN, kPair>;
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(block_threads<kGather>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!configured[d]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (kPair) {
      cfg.gridDim = dim3(2 * kMaxDevices);    // any even size: the query asks how many fit
      e = cudaOccupancyMaxActiveClusters(&max_pairs[d], kern, &cfg);
      if (e != cudaSuccess) return e;
      if (max_pairs[d] < 1) return cudaErrorInvalidConfiguration;
    }
    configured[d] = true;
  }
  if (!kPair) {
    kern<<<grid, block_threads<kGather>(), smem, st>>>(a, b0, b1, o.map[0], o.map[1], o.map[2], p);
    return cudaGetLastError();
  }
  // a persistent grid of pairs: at most one pair per two of the CTAs asked
  // for, and no more pairs than fit on the GPU at once
  const int pairs = grid / 2 < max_pairs[d] ? (grid / 2 > 0 ? grid / 2 : 1) : max_pairs[d];
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, kern, a, b0, b1, o.map[0], o.map[1], o.map[2], p);
}

template <Epi kEpi, bool kAmn, bool kBmn, Sched kSched, bool kGather = false>
cudaError_t launch_impl(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        const GemmOut& o, const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  if constexpr (!kGather && (kSched == Sched::Rows ? !kAmn : (kAmn && kBmn))) {
    if (p.pair) {
      if (kEpi == Epi::SwigluFwd || p.bn == 256)
        return launch_bn<kEpi, kAmn, kBmn, kSched, kGather, 256, true>(a, b0, b1, o, p, grid, st);
      return launch_bn<kEpi, kAmn, kBmn, kSched, kGather, 128, true>(a, b0, b1, o, p, grid, st);
    }
  }
  if (kEpi == Epi::SwigluFwd || p.bn == 256)
    return launch_bn<kEpi, kAmn, kBmn, kSched, kGather, 256, false>(a, b0, b1, o, p, grid, st);
  return launch_bn<kEpi, kAmn, kBmn, kSched, kGather, 128, false>(a, b0, b1, o, p, grid, st);
}

}  // namespace

cudaError_t launch_fc1_swiglu(const CUtensorMap& a, const CUtensorMap& wg, const CUtensorMap& wu,
                              const GemmOut& o, const GroupedGemmArgs& p, int grid,
                              cudaStream_t st) {
  return launch_impl<Epi::SwigluFwd, false, true, Sched::Rows>(a, wg, wu, o, p, grid, st);
}

cudaError_t launch_fc1_swiglu_gather(const CUtensorMap& x_rows, const CUtensorMap& wg,
                                     const CUtensorMap& wu, const GemmOut& o,
                                     const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  return launch_impl<Epi::SwigluFwd, false, true, Sched::Rows, true>(x_rows, wg, wu, o, p, grid,
                                                                     st);
}

cudaError_t launch_fc2(const CUtensorMap& a, const CUtensorMap& w, const GemmOut& o,
                       const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  return launch_impl<Epi::Bf16, false, true, Sched::Rows>(a, w, w, o, p, grid, st);
}

cudaError_t launch_dh_swiglu_bwd(const CUtensorMap& a, const CUtensorMap& w2, const GemmOut& o,
                                 const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  return launch_impl<Epi::SwigluBwd, false, false, Sched::Rows>(a, w2, w2, o, p, grid, st);
}

cudaError_t launch_dxp(const CUtensorMap& a, const CUtensorMap& wg, const CUtensorMap& wu,
                       const GemmOut& o, const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  return launch_impl<Epi::Bf16, false, false, Sched::Rows>(a, wg, wu, o, p, grid, st);
}

cudaError_t launch_wgrad(const CUtensorMap& a, const CUtensorMap& b, const GemmOut& o,
                         const GroupedGemmArgs& p, int grid, cudaStream_t st) {
  return launch_impl<Epi::F32, true, true, Sched::WGrad>(a, b, b, o, p, grid, st);
}

}  // namespace moe
