// gemm_mxfp8.cu - persistent grouped GEMMs of the MXFP8 expert block on the
// block-scaled tensor cores of sm_103a (tcgen05.mma.kind::mxf8f6f4 with one
// E8M0 scale per 32 elements of K on both operands), forward and backward.
//
// The structure is the one of gemm_bf16.cu (TMA producer warp, single-thread
// MMA issuer, TMEM accumulators, epilogue warps, a ring of `stages`
// shared-memory slots), with these differences:
//   * a k-block is 128 E4M3 elements (128 bytes, one 128B-swizzle row);
//     A (128 rows) and B (128 rows per box) are both K-major;
//   * the scales of a k-block, one 512-byte atom for A and one per 128 rows
//     of B, arrive by 1D bulk copies into the same slot and are moved into
//     tensor memory with tcgen05.cp (32x128b, replicated over the four lane
//     quadrants); each of the four MMAs of the k-block (K = 32) picks its
//     byte of the 32-bit scale words through the instruction's scale-factor id;
//   * slots are smaller than BF16 ones, so the ring is up to 6 deep: at the
//     FP8 rate 4 slots in flight per SM do not cover the L2 latency.
// Epilogues (MxEpi): fc1 rounds h to bf16 and quantises it per 32 along F
// (codes + tiled scales for fc2), optionally saving A_g, A_u and h in bf16
// for the backward; fc2 and dXp round their rows to bf16; dH applies the
// SwiGLU backward to the saved A_g, A_u; F32 writes weight-gradient rows
// (reduce-added when accumulating). Rows leave through per-warp shared-memory
// pieces and TMA tensor stores, except fc1's codes and scales and the bf16
// tensors kept in 32 x 32 blocks (fc1's saves, dH's dA), which are stored
// from registers. dH runs 12 warps with a register split (see reg_split).
// This is the quantised AllToAll+Matmul (MX FP8) of "MC2 通算融合架构总览",
// section 1, on one GPU, with its scales in buffers of their own (section 5).
// Schedules: Rows (expert segments padded to 128 rows; M fastest within an
// expert unless it has more M tiles than N tiles) and WGrad (K runs over one
// expert's padded rows; every expert owns M/128 x N/bn output tiles, the
// larger operand's dimension fastest, and an expert without rows writes
// zeros). CTA b takes tiles b,
// b + grid, ...
#include "common.cuh"
#include "internal.h"
#include "mx.cuh"

namespace moe {

namespace {

constexpr int BK = 128;                    // E4M3 elements (bytes) per k-block
constexpr int kABytes = kTileM * BK;       // 16 KB
constexpr int kSfBytes = 512;              // one scale atom (128 rows x 4 blocks of 32)
// warp 0 producer, warp 1 MMA issuer, then the epilogue warps. The fc1 and
// dH epilogues (SwiGLU forward + quantisation, SwiGLU backward) are heavy,
// and a float row of 256 columns does not fit one thread's registers: 8
// warps, two per TMEM lane quadrant, each finishing half of the tile's
// columns. fc2's bf16 row fits one thread: 4 warps (more only take issue
// slots from the producer and MMA threads).
template <MxEpi kEpi>
constexpr int epi_warps() { return kEpi == MxEpi::Bf16 ? 4 : 8; }
// dH also needs its float half-row (128 columns) next to the A_g, A_u blocks
// it reads, more than 168 registers a thread. Its CTA runs 12 warps: warps
// 0-3 (producer, MMA issuer and two idle warps that only complete the
// warpgroup) drop to kRegsControl registers, and the two epilogue
// warpgroups, warps 4-11, rise to kRegsEpi. setmaxnreg.inc waits until the
// CTA's pool (its registers at launch) has room, so the split must add up
// to exactly that pool: the launch checks the kernel's register count.
template <MxEpi kEpi>
constexpr bool reg_split() { return kEpi == MxEpi::SwigluBwd; }
template <MxEpi kEpi>
constexpr int epi_first_warp() { return reg_split<kEpi>() ? 4 : 2; }
template <MxEpi kEpi>
constexpr int num_threads() { return 32 * (epi_first_warp<kEpi>() + epi_warps<kEpi>()); }
constexpr int kRegsLaunch = 168;    // 65536 / 384 threads, in steps of 8
constexpr int kRegsControl = 56, kRegsEpi = 224;
static_assert(4 * kRegsControl + 8 * kRegsEpi == 12 * kRegsLaunch,
              "the register split must fill the pool of a 12-warp CTA exactly");

template <int kRegs>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <int kRegs>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kDrainNs = 1000000000ull;
constexpr unsigned long long kPairDrainNs = 50000000ull;

constexpr int kMaxStages = 8;

// Tile geometry for an MMA N of 128 or 256. N=128: two accumulators of 128
// columns (the epilogue of a tile overlaps the next tile) and 34 KB slots;
// N=256: one accumulator of 256 columns (no overlap, but half the A reads
// per FLOP) and 50 KB slots. Scales take 4 + N/32 columns per slot after the
// accumulators. A CTA of a pair (kPair, M = 256 over the two CTAs) holds
// half of the N tile's B rows but the scales of the whole N tile (its SM's
// tensor core scales all N columns of its own 128 rows): 34 KB slots, 6 of
// them, for N = 256; 25 KB slots, 8 of them, and two accumulators for
// N = 128, which streams as few operand bytes per SM and FLOP as one CTA
// with N = 256 while the epilogue of a tile overlaps the next one.
template <int kN, bool kPair = false>
struct MxGeo {
  static constexpr int kBBytes = (kPair ? kN / 2 : kN) * BK;
  static constexpr int kSfbAtoms = kN / 128;
  static constexpr int kStageBytes = ((kABytes + kBBytes + (1 + kSfbAtoms) * kSfBytes) + 1023) /
                                     1024 * 1024;
  static constexpr int kAccBufs = kN == 128 ? 2 : 1;
  static constexpr uint32_t kSfCol = kAccBufs * kN;
  static constexpr uint32_t kSfColsPerStage = 4 + 4 * kSfbAtoms;
  // what fits in shared memory
  static constexpr int kStages = kPair ? (kN == 128 ? 8 : 6) : (kN == 128 ? 6 : 4);
};

// Output rows leave as per-warp pieces of 32 rows x 64 bytes (32 bf16 or
// 16 float columns): each epilogue warp fills its own shared-memory slot,
// with the 64-byte swizzle of the output maps (16-byte chunk j of row r at
// chunk j ^ ((r >> 1) & 3)), and its lane 0 writes it with a TMA tensor
// store (or reduce-add). Whole-row bursts replace per-thread stores that
// would scatter 32 rows per warp instruction.
constexpr int kPieceBytes = 32 * 64;                  // 2 KB
constexpr int kPieceArea = 8 * kPieceBytes;           // one slot per epilogue warp

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

// One output tile: expert, M tile, N tile, its k-blocks and the first
// k-block's K offset (WGrad: the expert's first padded row).
struct MxTile {
  int e, m, n, kblocks, k0;
  int row0;        // Rows: first A row of the tile (of the pair's tile)
  int half_rows;   // pairs: 128-row blocks of the tile inside the expert (1 or 2)
};

template <MxEpi kEpi, Sched kSched, int kTileN, bool kPair>
__global__ void __launch_bounds__(num_threads<kEpi>(), 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmO0,
                   const __grid_constant__ CUtensorMap tmO1,
                   const __grid_constant__ CUtensorMap tmO2,
                   const __grid_constant__ CUtensorMap tmSA,
                   const __grid_constant__ CUtensorMap tmSB0,
                   const __grid_constant__ CUtensorMap tmSB1, MxGemmArgs p) {
  static_assert(!kPair || kSched == Sched::Rows, "CTA pairs run the Rows schedule");
  constexpr bool kFc1 = kEpi == MxEpi::Fc1 || kEpi == MxEpi::Fc1Save;
  constexpr bool kSave = kEpi == MxEpi::Fc1Save;   // fc1 also stores A_g, A_u and h in bf16
  constexpr bool kWGrad = kSched == Sched::WGrad;
  constexpr int kThreads = num_threads<kEpi>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using G = MxGeo<kTileN, kPair>;
  constexpr int kBBytes = G::kBBytes;
  constexpr int kStageBytes = G::kStageBytes;
  const int S = p.stages < G::kStages ? p.stages : G::kStages;
  uint8_t* pieces = ring + S * kStageBytes;
  Smem* sm = reinterpret_cast<Smem*>(pieces + kPieceArea);
  int* ts = reinterpret_cast<int*>(sm + 1);
  const int warp = threadIdx.x >> 5, lane = lane_id();
  const int E = p.E;
  const int n_cols = kFc1 ? kTileN / 2 : kTileN;   // output columns per N tile
  const int n_tiles = p.N / n_cols;
  const int kgroups_a = p.kgroups_a > 0 ? p.kgroups_a : (p.K >> 7);
  const int kgroups_b = p.kgroups_b > 0 ? p.kgroups_b : (p.K >> 7);
  const int m_tiles_w = kWGrad ? p.M / kTileM : 1;   // WGrad: M tiles of every expert
  // CTA pairs: this CTA's rank and the tile walk over clusters
  const uint32_t rank = kPair ? cluster_ctarank() : 0;
  const int walk0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int walk_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm->tfull[a]), 1);
      // one arrival per epilogue warp (of both CTAs of a pair)
      mbar_init(smem_u32(&sm->tempty[a]), (kPair ? 2 : 1) * epi_warps<kEpi>());
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
    if (kPair) {
      tmem_alloc_pair(smem_u32(&sm->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  if (!kWGrad) {
    for (int e = threadIdx.x; e < E; e += kThreads) {
      const int mb = (p.off_al[e + 1] - p.off_al[e]) / kTileM;
      ts[e + 1] = (kPair ? (mb + 1) >> 1 : mb) * n_tiles;
    }
  }
  __syncthreads();
  if (!kWGrad && threadIdx.x == 0) {
    ts[0] = 0;
    for (int e = 0; e < E; ++e) ts[e + 1] += ts[e];
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();   // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_base;
  const int total = kWGrad ? E * m_tiles_w * n_tiles : ts[E];
  volatile int* abort_flag = &sm->abort;

  auto decode = [&](int t) {
    MxTile tl;
    tl.half_rows = 1;
    tl.row0 = 0;
    if (kWGrad) {
      const int per = m_tiles_w * n_tiles;
      tl.e = t / per;
      const int local = t - tl.e * per;
      if (p.M > p.N) {        // A is the larger operand: N fastest keeps B's panels in L2
        tl.m = local / n_tiles;
        tl.n = local - tl.m * n_tiles;
      } else {                // B is larger: M fastest keeps A's panels in L2
        tl.n = local / m_tiles_w;
        tl.m = local - tl.n * m_tiles_w;
      }
      tl.k0 = p.off_al[tl.e];
      tl.kblocks = (p.off_al[tl.e + 1] - tl.k0) / BK;
      return tl;
    }
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ts[mid] <= t) lo = mid; else hi = mid - 1;
    }
    tl.e = lo;
    const int mb = (p.off_al[tl.e + 1] - p.off_al[tl.e]) / kTileM;
    const int mt = kPair ? (mb + 1) >> 1 : mb;
    const int local = t - ts[tl.e];
    if (mt > n_tiles) {       // tall expert: keep its row panel in L2
      tl.m = local / n_tiles;
      tl.n = local - tl.m * n_tiles;
    } else {
      tl.n = local / mt;
      tl.m = local - tl.n * mt;
    }
    tl.row0 = p.off_al[tl.e] + tl.m * (kPair ? 2 * kTileM : kTileM);
    if (kPair) tl.half_rows = min(2, mb - 2 * tl.m);
    tl.k0 = 0;
    tl.kblocks = p.K / BK;
    return tl;
  };

  // warpgroup-uniform role split: the register move, when there is one, is
  // the first thing each side runs, so all the code after it is compiled
  // against its new register count
  if (warp < epi_first_warp<kEpi>()) {
    if constexpr (reg_split<kEpi>()) regs_dec<kRegsControl>();
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t fills = 0;
        bool ok = true;
        const uint64_t pol_a = p.keep_a ? l2_policy_evict_last() : l2_policy_evict_normal();
        const uint64_t pol_b = l2_policy_evict_normal();
        const uint32_t ring0 = smem_u32(ring);
        for (int t = walk0; t < total && ok; t += walk_step) {
          const MxTile tl = decode(t);
          // A rows and the first 128-row block of B's scale atoms
          const int a_row = kWGrad ? tl.m * kTileM : tl.row0 + static_cast<int>(rank) * kTileM;
          const int64_t b_row =
              kWGrad ? static_cast<int64_t>(tl.n) * kTileN
                     : static_cast<int64_t>(tl.e) * p.b_rows + static_cast<int64_t>(tl.n) * (kFc1 ? kTileN / 2 : kTileN);
          const int64_t vrow = kWGrad ? b_row
                                      : static_cast<int64_t>(tl.e) * p.sfb_rows +
                                            static_cast<int64_t>(tl.n) * kTileN;
          const int kg0 = tl.k0 >> 7;
          // pairs: the second CTA's rows may lie past the expert (odd tail)
          const bool load_a = !kPair || static_cast<int>(rank) < tl.half_rows;
          for (int kb = 0; kb < tl.kblocks; ++kb) {
            const uint32_t full = smem_u32(&sm->full[stage]);
            if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.wait_ns, abort_flag)) {
              ok = false;
              break;
            }
            if constexpr (kPair) {
              // every copy of both CTAs completes on the leader's full barrier,
              // armed by the leader with the pair tile's bytes: A and its
              // scale atom per live half, both halves of B, and each CTA's
              // copy of the N tile's B scales
              const uint32_t full_l = mapa_shared(full, 0);
              if (rank == 0)
                mbar_arrive_expect_tx(full, tl.half_rows * (kABytes + kSfBytes) + kTileN * BK +
                                                2 * G::kSfbAtoms * kSfBytes);
              const uint32_t sa = ring0 + stage * kStageBytes;
              const uint32_t sb = sa + kABytes;
              const uint32_t ssf = sb + kBBytes;
              const int kx = kb * BK;
              const bool second = !kFc1 && p.k_split > 0 && kb >= p.k_split;
              const int kbb = second ? kb - p.k_split : kb;
              if (load_a) {
                tma_load_2d_pair(sa, &tmA, full_l, kx, a_row, pol_a);
                const int64_t atom = (static_cast<int64_t>(a_row) >> 7) * kgroups_a + kb;
                tma_load_2d_pair_plain(ssf, &tmSA, full_l, 0, static_cast<int>(2 * atom));
              }
              // this CTA's N / 2 rows of B (one box): fc1's gate rows (rank 0)
              // or up rows (rank 1), else its half of the N tile
              if (kFc1)
                tma_load_2d_pair(sb, rank == 0 ? &tmB0 : &tmB1, full_l, kx, static_cast<int>(b_row),
                                 pol_b);
              else
                tma_load_2d_pair(sb, second ? &tmB1 : &tmB0, full_l, kbb * BK,
                                 static_cast<int>(b_row) + static_cast<int>(rank) * (kTileN / 2),
                                 pol_b);
              const CUtensorMap* msb = second ? &tmSB1 : &tmSB0;
#pragma unroll
              for (int j = 0; j < G::kSfbAtoms; ++j)
                tma_load_2d_pair_plain(ssf + (1 + j) * kSfBytes, msb, full_l, 0,
                                       static_cast<int>(2 * (((vrow >> 7) + j) * kgroups_b + kbb)));
              ++fills;
              if (++stage == S) {
                stage = 0;
                phase ^= 1;
              }
              continue;
            }
            mbar_arrive_expect_tx(full, kABytes + kBBytes + (1 + G::kSfbAtoms) * kSfBytes);
            const uint32_t sa = ring0 + stage * kStageBytes;
            const uint32_t sb = sa + kABytes;
            const uint32_t ssf = sb + kBBytes;
            const int kx = tl.k0 + kb * BK;
            tma_load_2d_hint(sa, &tmA, full, kx, a_row, pol_a);
            // B: fc1 takes N/2 gate rows and N/2 up rows of the same N tile;
            // a K-split GEMM takes its k-blocks from B0, then from B1
            const bool second = !kFc1 && !kWGrad && p.k_split > 0 && kb >= p.k_split;
            const int kbb = second ? kb - p.k_split : kb;
            if (kFc1) {
              const int half = kTileN / 2;
              tma_load_2d(sb, &tmB0, full, kx, static_cast<int>(b_row));
              tma_load_2d(sb + half * BK, &tmB1, full, kx, static_cast<int>(b_row));
            } else {
              const CUtensorMap* mb = second ? &tmB1 : &tmB0;
              for (int j = 0; j < kTileN; j += 128)
                tma_load_2d(sb + j * BK, mb, full, kbb * BK + tl.k0, static_cast<int>(b_row + j));
            }
            // the scale atoms through the 2D scale maps (one atom per box): a
            // plain bulk copy holds the issuing thread for about as long as its
            // bytes take to arrive, a tensor-map copy does not
            tma_load_2d(ssf, &tmSA, full, 0,
                        static_cast<int>(2 * ((static_cast<int64_t>(a_row) >> 7) * kgroups_a + kg0 + kb)));
            const CUtensorMap* msb = second ? &tmSB1 : &tmSB0;
#pragma unroll
            for (int j = 0; j < G::kSfbAtoms; ++j)
              tma_load_2d(ssf + (1 + j) * kSfBytes, msb, full, 0,
                          static_cast<int>(2 * (((vrow >> 7) + j) * kgroups_b + kg0 + kbb)));
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
        // the last S fills must land before exit (fill i: slot i % S, parity
        // (i / S) & 1). A pair's copies complete on the leader's barrier: each
        // CTA waits until the MMAs that read its last fills released them,
        // briefly after an abort, when they may never come (a copy lands
        // within microseconds).
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
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true, issued = false;
        for (int t = walk0; t < total && ok; t += walk_step) {
          const int kblocks = decode(t).kblocks;
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
            const uint64_t ad = sdesc_sw128(sa, 16, 1024), bd = sdesc_sw128(sb, 16, 1024);
            if constexpr (kPair) {
              tmem_cp_32x128b_warpx4_pair(sfa_t, sdesc_noswizzle(ssf, 16, 128));
#pragma unroll
              for (int j = 0; j < G::kSfbAtoms; ++j)
                tmem_cp_32x128b_warpx4_pair(sfb_t + 4 * j,
                                            sdesc_noswizzle(ssf + (1 + j) * kSfBytes, 16, 128));
#pragma unroll
              for (int ks = 0; ks < BK / 32; ++ks)
                umma_mxf8_pair(d, ad + 2 * ks, bd + 2 * ks, idesc_mxf8(2 * kTileM, kTileN, ks, ks),
                               sfa_t, sfb_t, (kb | ks) ? 1u : 0u);
              umma_commit_pair_mc(smem_u32(&sm->empty[stage]), 0x3);   // the slot, in both CTAs
            } else {
              tmem_cp_32x128b_warpx4(sfa_t, sdesc_noswizzle(ssf, 16, 128));
#pragma unroll
              for (int j = 0; j < G::kSfbAtoms; ++j)
                tmem_cp_32x128b_warpx4(sfb_t + 4 * j,
                                       sdesc_noswizzle(ssf + (1 + j) * kSfBytes, 16, 128));
#pragma unroll
              for (int ks = 0; ks < BK / 32; ++ks)      // +32 B of K per MMA
                umma_mxf8(d, ad + 2 * ks, bd + 2 * ks, idesc_mxf8(kTileM, kTileN, ks, ks), sfa_t,
                          sfb_t, (kb | ks) ? 1u : 0u);
              umma_commit(smem_u32(&sm->empty[stage]));
            }
            issued = true;
            if (++stage == S) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          // a tile without k-blocks (WGrad, an expert without rows) issued no
          // MMA: the commit only hands the (unwritten) accumulator on
          if (kPair)
            umma_commit_pair_mc(smem_u32(&sm->tfull[acc]), 0x3);   // both CTAs' epilogues
          else
            umma_commit(smem_u32(&sm->tfull[acc]));
          issued = true;
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
          if (kPair)
            umma_commit_pair_mc(smem_u32(&sm->drain), 0x1);
          else
            umma_commit(smem_u32(&sm->drain));
          mbar_wait(smem_u32(&sm->drain), 0, kDrainNs, &sm->zero);
        }
      }
    }      // warps 2 and 3 of a 12-warp CTA have no role
  } else {
    if constexpr (reg_split<kEpi>()) regs_inc<kRegsEpi>();
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;                   // TMEM lane quadrant of this warp
    const int ew = warp - epi_first_warp<kEpi>();
    const int half = ew >> 2;                 // 8 warps: which half of the tile's columns
    const int row_in_tile = q * 32 + lane;
    // 8 slots in all: one per warp of an 8-warp epilogue, two (alternating)
    // per warp of a 4-warp one
    constexpr int kSlots = 8 / epi_warps<kEpi>();
    const uint32_t slot0 = smem_u32(pieces) + ew * kSlots * kPieceBytes;
    const uint32_t my_row = lane * 64;
    const uint32_t sw = (lane >> 1) & 3;
    int npiece = 0;
    // a piece: wait until the warp's next slot has been read by its last
    // store, fill this lane's 64-byte row, hand the slot to TMA
    auto put_piece = [&](const uint32_t* w16, const CUtensorMap* map, int x, int y, bool add) {
      if (lane == 0) bulk_wait_group_read<kSlots - 1>();
      __syncwarp();
      const uint32_t slot = slot0 + (npiece % kSlots) * kPieceBytes;
      ++npiece;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(slot + my_row +
                                                                       ((j ^ sw) << 4)),
                     "r"(w16[4 * j]), "r"(w16[4 * j + 1]), "r"(w16[4 * j + 2]),
                     "r"(w16[4 * j + 3])
                     : "memory");
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        if (add) tma_reduce_add_2d(map, slot, x, y);
        else tma_store_2d(map, slot, x, y);
        bulk_commit_group();
      }
    };
    // a 32 x 32 bf16 block of A_g or A_u in the blocked layout
    // (act_block_offset): lane r's row is its four 16-byte slab pieces, so
    // each warp store writes 512 contiguous bytes straight from registers
    auto put_block = [&](const uint32_t* w16, __nv_bfloat16* dst) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_global_v4(dst + j * 256 + lane * 8, w16[4 * j], w16[4 * j + 1], w16[4 * j + 2],
                     w16[4 * j + 3]);
    };
    auto bf16_words = [](const uint32_t* f32x32, uint32_t* w16) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w16[i] = pack_bf16x2(__uint_as_float(f32x32[2 * i]), __uint_as_float(f32x32[2 * i + 1]));
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    // the accumulator is handed back to the MMA issuer (the leader, for a
    // pair) by one arrival per warp, once the warp's reads of it are done
    const uint32_t tempty0 = kPair ? mapa_shared(smem_u32(&sm->tempty[0]), 0) : 0;
    auto release_acc = [&](int a) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair)
          mbar_arrive_cluster(tempty0 + a * static_cast<uint32_t>(sizeof(uint64_t)));
        else
          mbar_arrive(smem_u32(&sm->tempty[a]));
      }
    };
    for (int t = walk0; t < total; t += walk_step) {
      const MxTile tl = decode(t);
      // this CTA's 128 rows of the tile; pairs: rows past the expert are not live
      const int my_row0 = tl.row0 + static_cast<int>(rank) * kTileM;
      const bool live = !kPair || static_cast<int>(rank) < tl.half_rows;
      const int64_t grow = kWGrad ? 0 : my_row0 + row_in_tile;
      const int wrow0 = kWGrad ? 0 : my_row0 + q * 32;   // warp's first row
      // SwigluBwd: this row's A_g, A_u over the warp's half of the tile, 32
      // columns at a time as packed bf16 pairs, from the blocked layout (four
      // coalesced 512-byte loads per 32 x 32 block). The first block of each
      // arrives while the tile's MMAs run; the rest are brought into L2 now
      // and into registers one step ahead of their use.
      constexpr int kActW = 16;                  // words of 32 columns
      uint32_t ag_w[kActW], au_w[kActW];
      const int act_c0 = tl.n * kTileN + half * (kTileN / 2);
      auto act_block = [&](const __nv_bfloat16* act, int c) {   // this lane's row of a block
        return act + act_block_offset(wrow0, act_c0 + c, p.N) + lane * 8;
      };
      auto load_act = [&](const __nv_bfloat16* row, uint32_t* w16) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int4 v = __ldg(reinterpret_cast<const int4*>(row + j * 256));
          w16[4 * j] = static_cast<uint32_t>(v.x);
          w16[4 * j + 1] = static_cast<uint32_t>(v.y);
          w16[4 * j + 2] = static_cast<uint32_t>(v.z);
          w16[4 * j + 3] = static_cast<uint32_t>(v.w);
        }
      };
      if (kEpi == MxEpi::SwigluBwd && live) {
#pragma unroll
        for (int c = 32; c < kTileN / 2; c += 32)   // 16 lines per block: lanes 0-15 A_g
          prefetch_l2(act_block(lane < 16 ? p.act_g : p.act_u, c) - lane * 8 + (lane & 15) * 64);
        load_act(act_block(p.act_g, 0), ag_w);
        load_act(act_block(p.act_u, 0), au_w);
      }
      const bool got = mbar_wait(smem_u32(&sm->tfull[acc]), acc_phase, p.wait_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        sm->abort = 1;
        if (lane == 0) report_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kTileN;
      if (!live) {
        release_acc(acc);   // pairs: rows past the expert; nothing to keep
      } else if (kFc1) {
        // h = bf16(silu(gate) * up), then MXFP8 per 32 along F. h is held
        // packed in bf16 (it is bf16-valued, so nothing is lost) and the
        // accumulator is released before the quantisation and the stores,
        // which then overlap the next tile's MMAs. The tile's N/64 scale
        // bytes of this row are adjacent in the tiled layout (one 128-wide K
        // group of fc2): they leave in one store. With save, A_g and A_u are
        // packed too, and A_g, A_u and h leave in bf16 after the release, in
        // the blocked layout, straight from registers. This warp's half of
        // the tile's h columns: kTileN / 4.
        constexpr int kHalf = kTileN / 4;
        const int c0 = half * kHalf;
        const int col = tl.n * n_cols + c0;
        uint32_t hw[kHalf / 2];
        uint32_t gw[kHalf / 2], uw[kHalf / 2];    // with save: A_g, A_u packed
        auto h_pair = [](uint32_t g0, uint32_t g1, uint32_t u0, uint32_t u1) {
          return pack_bf16x2(silu_f(__uint_as_float(g0)) * __uint_as_float(u0),
                             silu_f(__uint_as_float(g1)) * __uint_as_float(u1));
        };
        if (kSave) {
#pragma unroll
          for (int c = 0; c < kHalf; c += 16) {   // 16 columns at a time: few live registers
            uint32_t g[16], u[16];
            tmem_ld_32x32b_x16(taddr + c0 + c, g);
            tmem_ld_32x32b_x16(taddr + kTileN / 2 + c0 + c, u);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              hw[c / 2 + i] = h_pair(g[2 * i], g[2 * i + 1], u[2 * i], u[2 * i + 1]);
              gw[c / 2 + i] = pack_bf16x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
              uw[c / 2 + i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < kHalf; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(taddr + c0 + c, g);
            tmem_ld_32x32b_x32(taddr + kTileN / 2 + c0 + c, u);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              hw[c / 2 + i] = h_pair(g[2 * i], g[2 * i + 1], u[2 * i], u[2 * i + 1]);
          }
        }
        release_acc(acc);
        if (kSave) {                               // after the release: off the MMAs' path
#pragma unroll
          for (int c = 0; c < kHalf; c += 32) {
            put_block(&gw[c / 2], p.save_g + act_block_offset(wrow0, col + c, p.N));
            put_block(&uw[c / 2], p.save_u + act_block_offset(wrow0, col + c, p.N));
            put_block(&hw[c / 2], p.save_h + act_block_offset(wrow0, col + c, p.N));
          }
        }
        uint32_t codes[kHalf / 4];
        uint32_t packed = 0;
#pragma unroll
        for (int c = 0; c < kHalf; c += 32) {
          float hv[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[c / 2 + i]));
            hv[2 * i] = f.x;
            hv[2 * i + 1] = f.y;
          }
          const uint8_t sc = quantize_block32(hv, &hw[c / 2], &codes[c / 4]);
          packed |= static_cast<uint32_t>(sc) << (8 * (c >> 5));
        }
        int4* dst = reinterpret_cast<int4*>(p.hq + grow * p.N + col);
#pragma unroll
        for (int i = 0; i < kHalf / 16; ++i)
          dst[i] = make_int4(codes[4 * i], codes[4 * i + 1], codes[4 * i + 2], codes[4 * i + 3]);
        uint8_t* hs = p.hs + mx_scale_offset(grow, col >> 5, p.N);
        if (kHalf == 64)
          *reinterpret_cast<uint16_t*>(hs) = static_cast<uint16_t>(packed);
        else
          *hs = static_cast<uint8_t>(packed);
      } else if (kEpi == MxEpi::Bf16) {
        // O = bf16: the row is packed into registers and the accumulator
        // released before its pieces (32 columns each) go out
        uint32_t w[kTileN / 2];
#pragma unroll
        for (int c = 0; c < kTileN; c += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c, r);
          tmem_ld_wait();
          bf16_words(r, &w[c / 2]);
        }
        release_acc(acc);
#pragma unroll
        for (int c = 0; c < kTileN; c += 32)
          put_piece(&w[c / 2], &tmO0, tl.n * kTileN + c, wrow0, false);
      } else if (kEpi == MxEpi::SwigluBwd) {
        // dA_g = bf16(dH A_u s (1 + A_g (1 - s))), dA_u = bf16(dH A_g s),
        // s = sigmoid(A_g), over this warp's half of the tile's columns; dA_g
        // at column f of [dA_g | dA_u], dA_u at N + f, in the blocked layout
        // (the dual quantiser reads it), straight from registers. The warp's
        // whole half-row of dH is loaded and the accumulator released first,
        // so the next tile's MMAs run under this arithmetic and these stores.
        constexpr int kHalf = kTileN / 2;
        const int f0 = tl.n * kTileN + half * kHalf;
        uint32_t v[kHalf];
#pragma unroll
        for (int c = 0; c < kHalf; c += 32) tmem_ld_32x32b_x32(taddr + half * kHalf + c, &v[c]);
        tmem_ld_wait();
        release_acc(acc);
#pragma unroll
        for (int c = 0; c < kHalf; c += 32) {
          uint32_t ag_n[kActW], au_n[kActW];      // the next 32 columns, in flight
          if (c + 32 < kHalf) {
            load_act(act_block(p.act_g, c + 32), ag_n);
            load_act(act_block(p.act_u, c + 32), au_n);
          }
          uint32_t wg[16], wu[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float vg[2], vu[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float dh = __uint_as_float(v[c + 2 * i + h]);
              const float a = __uint_as_float(h ? (ag_w[i] & 0xFFFF0000u) : (ag_w[i] << 16));
              const float b = __uint_as_float(h ? (au_w[i] & 0xFFFF0000u) : (au_w[i] << 16));
              const float sg = sigmoid_f(a);
              vg[h] = dh * b * sg * (1.0f + a * (1.0f - sg));
              vu[h] = dh * a * sg;
            }
            wg[i] = pack_bf16x2(vg[0], vg[1]);
            wu[i] = pack_bf16x2(vu[0], vu[1]);
          }
          put_block(wg, p.out_b + act_block_offset(wrow0, f0 + c, 2 * p.N));
          put_block(wu, p.out_b + act_block_offset(wrow0, p.N + f0 + c, 2 * p.N));
          if (c + 32 < kHalf) {
#pragma unroll
            for (int i = 0; i < kActW; ++i) {
              ag_w[i] = ag_n[i];
              au_w[i] = au_n[i];
            }
          }
        }
      } else {
        // float rows, 16 columns per piece: a weight-gradient row (WGrad;
        // the expert's rows below out_split go to map 0 at row
        // e * out_split + r, the rest to map 1 at e * (M - out_split) + r -
        // out_split; out_split is a multiple of 128, so a tile is on one side)
        const CUtensorMap* map = &tmO0;
        int y = wrow0;
        if (kWGrad) {
          const int r = tl.m * kTileM + q * 32;
          const int split = p.out_split > 0 ? p.out_split : p.M;
          if (r < split) {
            y = tl.e * split + r;
          } else {
            map = &tmO1;
            y = tl.e * (p.M - split) + (r - split);
          }
        }
        const bool empty = tl.kblocks == 0;     // WGrad: an expert without rows
        const bool add = kWGrad && p.accumulate != 0;
        // this warp's half of the row, in registers, so that the
        // accumulator is released before the pieces go out
        constexpr int kCols = kTileN / 2;
        const int cbase = half * kCols;
        uint32_t v[kCols];
        if (!empty) {
#pragma unroll
          for (int c = 0; c < kCols; c += 32) tmem_ld_32x32b_x32(taddr + cbase + c, &v[c]);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < kCols; ++i) v[i] = 0u;
        }
        release_acc(acc);
        if (!(empty && add)) {
#pragma unroll
          for (int c = 0; c < kCols; c += 16)
            put_piece(&v[c], map, tl.n * kTileN + cbase + c, y, add);
        }
      }
      if (++acc == G::kAccBufs) {
        acc = 0;
        acc_phase ^= 1;
      }
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

template <MxEpi kEpi, Sched kSched, int kN, bool kPair>
cudaError_t launch_mx(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                      const GemmOut& o, const MxScaleMaps& sc, const MxGemmArgs& p, int grid,
                      cudaStream_t st) {
  using G = MxGeo<kN, kPair>;
  constexpr size_t smem = 1024 + G::kStages * static_cast<size_t>(G::kStageBytes) + kPieceArea +
                          sizeof(Smem) + static_cast<size_t>(kMaxExperts + 1) * sizeof(int);
  static_assert(smem <= 232448, "shared memory of one CTA");
  static_assert(G::kSfCol + G::kStages * G::kSfColsPerStage <= kTmemCols,
                "accumulators and scale columns fit the tensor memory");
  static bool configured[kMaxDevices] = {};    // the attribute is per device
  static int max_pairs[kMaxDevices] = {};      // clusters of two that fit at once
  auto kern = mx_gemm_kernel<kEpi, kSched, kN, kPair>;
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(num_threads<kEpi>());
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
    if (reg_split<kEpi>()) {
      // the split's setmaxnreg.inc would wait for good on a smaller pool
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
    }
    if (kPair) {
      cfg.gridDim = dim3(2 * kMaxDevices);    // any even size: the query asks how many fit
      e = cudaOccupancyMaxActiveClusters(&max_pairs[d], kern, &cfg);
      if (e != cudaSuccess) return e;
      if (max_pairs[d] < 1) return cudaErrorInvalidConfiguration;
    }
    configured[d] = true;
  }
  if (!kPair) {
    kern<<<grid, num_threads<kEpi>(), smem, st>>>(a, b0, b1, o.map[0], o.map[1], o.map[2],
                                                    sc.map[0], sc.map[1], sc.map[2], p);
    return cudaGetLastError();
  }
  const int pairs = grid / 2 < max_pairs[d] ? (grid / 2 > 0 ? grid / 2 : 1) : max_pairs[d];
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, kern, a, b0, b1, o.map[0], o.map[1], o.map[2], sc.map[0],
                            sc.map[1], sc.map[2], p);
}

// CTA pairs run tiles of the Rows schedule when asked for (a pair's B maps
// then have boxes of N / 2 rows); everything else runs one CTA per tile.
template <MxEpi kEpi, Sched kSched>
cudaError_t launch_mx_bn(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                         const GemmOut& o, const MxGemmArgs& p, int grid, cudaStream_t st,
                         const MxScaleMaps& sc) {
  if constexpr (kSched == Sched::Rows) {
    if (p.pair)
      return p.bn == 256 ? launch_mx<kEpi, kSched, 256, true>(a, b0, b1, o, sc, p, grid, st)
                         : launch_mx<kEpi, kSched, 128, true>(a, b0, b1, o, sc, p, grid, st);
  }
  return p.bn == 256 ? launch_mx<kEpi, kSched, 256, false>(a, b0, b1, o, sc, p, grid, st)
                     : launch_mx<kEpi, kSched, 128, false>(a, b0, b1, o, sc, p, grid, st);
}

}  // namespace

cudaError_t launch_mx_fc1(const CUtensorMap& a, const CUtensorMap& wg, const CUtensorMap& wu,
                          const GemmOut& o, const MxGemmArgs& p, int grid, cudaStream_t st,
                          const MxScaleMaps& sc) {
  return p.save ? launch_mx_bn<MxEpi::Fc1Save, Sched::Rows>(a, wg, wu, o, p, grid, st, sc)
                : launch_mx_bn<MxEpi::Fc1, Sched::Rows>(a, wg, wu, o, p, grid, st, sc);
}

cudaError_t launch_mx_fc2(const CUtensorMap& a, const CUtensorMap& wd, const GemmOut& o,
                          const MxGemmArgs& p, int grid, cudaStream_t st, const MxScaleMaps& sc) {
  return launch_mx_bn<MxEpi::Bf16, Sched::Rows>(a, wd, wd, o, p, grid, st, sc);
}

cudaError_t launch_mx_dh(const CUtensorMap& a, const CUtensorMap& w2, const GemmOut& o,
                         const MxGemmArgs& p, int grid, cudaStream_t st, const MxScaleMaps& sc) {
  return launch_mx_bn<MxEpi::SwigluBwd, Sched::Rows>(a, w2, w2, o, p, grid, st, sc);
}

cudaError_t launch_mx_dxp(const CUtensorMap& a, const CUtensorMap& w1g, const CUtensorMap& w1u,
                          const GemmOut& o, const MxGemmArgs& p, int grid, cudaStream_t st,
                          const MxScaleMaps& sc) {
  return launch_mx_bn<MxEpi::Bf16, Sched::Rows>(a, w1g, w1u, o, p, grid, st, sc);
}

cudaError_t launch_mx_wgrad(const CUtensorMap& a, const CUtensorMap& b, const GemmOut& o,
                            const MxGemmArgs& p, int grid, cudaStream_t st, const MxScaleMaps& sc) {
  return launch_mx_bn<MxEpi::F32, Sched::WGrad>(a, b, b, o, p, grid, st, sc);
}

}  // namespace moe
