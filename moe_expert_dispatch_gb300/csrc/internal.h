// internal.h - launchers shared between the translation units of the
// library. Nothing here is part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// An NVTX range named after the entry point around each C-ABI call, so that
// a profiler's timeline groups every launch under the call that made it.
// Without a tool attached a push or pop costs a few nanoseconds.
struct ScopedRange {
  explicit ScopedRange(const char* name) { nvtxRangePushA(name); }
  ~ScopedRange() { nvtxRangePop(); }
  ScopedRange(const ScopedRange&) = delete;
  ScopedRange& operator=(const ScopedRange&) = delete;
};
#define MOE_ENTRY_RANGE() ::moe::ScopedRange moe_entry_range_(__func__)

// Ids handled by one CTA of the histogram and row-map kernels.
constexpr int kRouteChunk = 2048;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
// Rows of one grouped-GEMM M tile; expert segments are padded to it.
constexpr int kTileM = 128;

inline int64_t route_chunks(int64_t n_ids) { return (n_ids + kRouteChunk - 1) / kRouteChunk; }

// Scratch of the counting step: per-chunk histograms and per-chunk bases,
// each [chunks, E] int32, after a 256-byte head whose first word is the
// completion ticket of the fused gate (route_topk); the head and the
// histograms are contiguous so that one memset clears both.
constexpr size_t kRouteHeadBytes = 256;
struct RouteScratch {
  int32_t* hist = nullptr;
  int32_t* base = nullptr;
  int64_t chunks = 0;
  unsigned int* ticket = nullptr;
};
size_t route_scratch_bytes(int64_t n_ids, int E);
RouteScratch route_scratch(void* ws, int64_t n_ids, int E);

// counts[E], offsets[E+1] (dense) and, when off_al != nullptr, the offsets
// of expert segments padded to `align` rows; s.base receives for every chunk
// and expert the first row its ids take (in the padded layout).
cudaError_t launch_counts(const int32_t* ids, int64_t n, int E, int align, int32_t* counts,
                          int32_t* offsets, int32_t* off_al, RouteScratch s, int* err,
                          cudaStream_t st);

// The gate ahead of the block from float logits [T, E]: ids[t] = the k
// largest logits in descending order (ties to the lower index, NaN as
// -inf), probs[t] = softmax over the chosen k; then, in the same launch,
// counts, offsets (and off_al, s.base as launch_counts). Clears the ticket
// and histograms of s itself (one memset).
cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int align,
                              int32_t* ids, float* probs, int32_t* counts, int32_t* offsets,
                              int32_t* off_al, RouteScratch s, cudaStream_t st);

// Row of every slot, token and prob of every row (stable within an expert).
// n_rows, err (here and below): the rows of the row-indexed buffers and the
// error word, for the bounds checks of the MOE_DEBUG build (n_rows < 0: none).
cudaError_t launch_rowmap(const int32_t* ids, const float* probs, int64_t n, int k, int E,
                          RouteScratch s, int32_t* row_of, int32_t* token_of, float* prob_of,
                          cudaStream_t st, int64_t n_rows = -1, int* err = nullptr);

// xp[row_of[t, j]] = x[t] for every token (rows of row_bytes, % 16 == 0).
cudaError_t launch_permute_copy(const void* x, int64_t T, int64_t row_bytes, int k,
                                const int32_t* row_of, void* xp, cudaStream_t st,
                                int64_t n_rows = -1, int* err = nullptr);

// Zero the padding rows of every expert segment of xp (and mark them in
// token_of / prob_of with -1 / 0).
cudaError_t launch_zero_padding(const int32_t* counts, const int32_t* off_al, int E,
                                int64_t row_bytes, void* xp, int32_t* token_of, float* prob_of,
                                cudaStream_t st);

cudaError_t launch_unpermute(const __nv_bfloat16* o, const int32_t* row_of, const float* probs,
                             int64_t T, int k, int H, __nv_bfloat16* y, cudaStream_t st,
                             int64_t n_rows = -1, int* err = nullptr);

cudaError_t launch_quantize_mxfp8(const __nv_bfloat16* in, int64_t rows, int K, uint8_t* q,
                                  uint8_t* scales, cudaStream_t st);
// The same with the scales in the MMA's tiled layout (rows % 128 == 0,
// K % 128 == 0); rows at or past *row_end (when given) are skipped.
cudaError_t launch_quantize_mxfp8_tiled(const __nv_bfloat16* in, int64_t rows, int K,
                                        const int32_t* row_end, uint8_t* q, uint8_t* scales,
                                        cudaStream_t st);
// Quantisation along the rows of in[z] [rows, cols] (z < batch; element
// (r, c) at in + z * batch_stride + r * ld + c): q[z] [cols, rows] codes,
// scales row-major [batch, cols, rows/32] or tiled for batch * cols rows and
// K = rows. rows % 32 == 0, cols % 8 == 0, ld % 8 == 0 (tiled: batch * cols
// % 128 == 0, rows % 128 == 0). With
// gather, row r reads row gather[r] of in (zero when outside [0, src_rows));
// row blocks at or past *row_end (when given) are skipped.
// Both orientations of in[z] [rows, cols] from one read: q_row [batch * rows,
// cols] along the columns (scales [batch * rows, cols/32], or tiled with
// K = cols) and q_col as launch_quantize_cols. rows % 32 == 0, cols % 128 == 0.
cudaError_t launch_quantize_dual(const __nv_bfloat16* in, int64_t ld, int64_t batch,
                                 int64_t batch_stride, int rows, int cols,
                                 const int32_t* row_end, bool tiled, uint8_t* q_row,
                                 uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                 cudaStream_t st);
cudaError_t launch_quantize_cols(const __nv_bfloat16* in, int64_t ld, int64_t batch,
                                 int64_t batch_stride, int rows, int cols, const int32_t* gather,
                                 int64_t src_rows, const int32_t* row_end, bool tiled, uint8_t* q,
                                 uint8_t* scales, cudaStream_t st);
// The same two quantisers, tiled scales, reading in [rows, cols] from the
// 32 x 32 blocked layout of act_block_offset (N = cols): rows % 32 == 0,
// cols % 128 == 0.
cudaError_t launch_quantize_dual_blocked(const __nv_bfloat16* in, int rows, int cols,
                                         const int32_t* row_end, uint8_t* q_row, uint8_t* s_row,
                                         uint8_t* q_col, uint8_t* s_col, cudaStream_t st);
cudaError_t launch_quantize_cols_blocked(const __nv_bfloat16* in, int rows, int cols,
                                         const int32_t* row_end, uint8_t* q, uint8_t* scales,
                                         cudaStream_t st);

// ------------------------------------------------------------------ grouped GEMMs

// Epilogue of a grouped GEMM.
enum class Epi {
  SwigluFwd,  // fc1: out = bf16(silu(gate) * up); gate/up are the two halves of the N tile
  Bf16,       // out = bf16(acc)
  SwigluBwd,  // dH -> dA_g, dA_u (bf16) from the saved A_g, A_u
  F32,        // float output: weight gradients (WGrad), optionally accumulated
};
// Tile schedule: M tiles over the routed rows of each expert (fixed K), or
// over the rows of each expert's weight gradient (K = the expert's rows).
enum class Sched { Rows, WGrad };

struct GroupedGemmArgs {
  const int32_t* off_al;   // [E+1] expert row offsets, multiples of kTileM
  int E;
  int K;                   // Rows: reduction length
  int M;                   // WGrad: rows of one expert's output (H or F)
  int N;                   // output columns (logical)
  int bn;                  // MMA N: 128 or 256
  int stages;              // ring depth 1..4
  int64_t b_rows;          // rows of one expert in B's 2D view
  int b_split;             // 0; 1: N tile = [B0 cols | B1 cols] (gate | up); 2: K split at k_split
  int k_split;             // k-blocks read from B0 when b_split == 2
  __nv_bfloat16* out;      // bf16 output
  int64_t ldo;             // row stride of out (elements)
  __nv_bfloat16* save_g;   // fc1: optional bf16 copy of A_g, blocked (act_block_offset)
  __nv_bfloat16* save_u;   // fc1: optional bf16 copy of A_u, blocked
  const __nv_bfloat16* act_g;  // SwigluBwd: saved A_g, blocked
  const __nv_bfloat16* act_u;  // SwigluBwd: saved A_u, blocked
  int64_t ld_act;          // columns of the saved A_g, A_u (F)
  int out_split;           // SwigluBwd: column offset of dA_u in out; F32: columns of outf
  float* outf;             // F32 output: Rows [rows, ldo]; WGrad [E, M, N or out_split]
  float* outf2;            // F32 second output (columns >= out_split)
  int accumulate;          // F32: add to the existing values
  int keep_a;              // L2 evict_last hint on A loads (A small enough to stay resident)
  const int32_t* gather_token;  // fc1 with fused gather: token of each padded row
  const int32_t* counts;        // fc1 with fused gather: rows of each expert
  const __nv_bfloat16* gather_x;  // fc1 with fused gather: x [T, K], rows read by cp.async
  int pair;                // Rows: CTA pairs (cta_group::2) share M = 256 tiles; a
                           // K-major B map then has boxes of bn/2 rows
  int* err;
  unsigned long long wait_ns;
};

// Encodes a 2D bf16 tensor map with the 128-byte swizzle (box inner = 64).
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// Output tensor maps of a grouped GEMM's epilogue: boxes of 32 rows x 64
// bytes with the 64-byte swizzle (see make_out_tmap). Unused maps may repeat
// a used one.
struct GemmOut {
  CUtensorMap map[3];
};
// A 2D output map over a row-major [outer, inner] tensor of bf16 (f32 = false)
// or float elements.
bool make_out_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, bool f32);

// fc1: out = bf16(silu(A W_gate) * (A W_up)), A rows tiled per expert.
// Outputs: h (map 0) and, with save_g, A_g and A_u as blocks (save_g, save_u).
cudaError_t launch_fc1_swiglu(const CUtensorMap& a, const CUtensorMap& wg, const CUtensorMap& wu,
                              const GemmOut& o, const GroupedGemmArgs& p, int grid,
                              cudaStream_t st);
// fc1 with the dispatch fused into its producer: A rows are gathered from
// the token rows of x (tensor map with a one-row box) by TMA gather4.
cudaError_t launch_fc1_swiglu_gather(const CUtensorMap& x_rows, const CUtensorMap& wg,
                                     const CUtensorMap& wu, const GemmOut& o,
                                     const GroupedGemmArgs& p, int grid, cudaStream_t st);
// fc2: out = bf16(A W) (map 0).
cudaError_t launch_fc2(const CUtensorMap& a, const CUtensorMap& w, const GemmOut& o,
                       const GroupedGemmArgs& p, int grid, cudaStream_t st);
// backward: dH = dO W2^T with the SwiGLU-backward epilogue (W2 read K-major);
// dA_g and dA_u into one [rows, 2F] tensor (map 0, columns [0, F) and [F, 2F)).
cudaError_t launch_dh_swiglu_bwd(const CUtensorMap& a, const CUtensorMap& w2, const GemmOut& o,
                                 const GroupedGemmArgs& p, int grid, cudaStream_t st);
// backward: dXp = bf16([dA_g | dA_u] [W1g ; W1u]^T) (K split between the two weights).
cudaError_t launch_dxp(const CUtensorMap& a, const CUtensorMap& wg, const CUtensorMap& wu,
                       const GemmOut& o, const GroupedGemmArgs& p, int grid, cudaStream_t st);
// backward: dW_e = A_e^T B_e over each expert's rows, both operands MN-major;
// float rows of [E*M, N] (map 0; map 1 for columns >= out_split), stored or,
// with accumulate, added (TMA reduce-add).
cudaError_t launch_wgrad(const CUtensorMap& a, const CUtensorMap& b, const GemmOut& o,
                         const GroupedGemmArgs& p, int grid, cudaStream_t st);

// backward: dO[r] = bf16(prob_of[r] dY[token_of[r]]) and dprobs[t, j] = <dY_t, O[row_of[t, j]]>.
cudaError_t launch_dout(const __nv_bfloat16* dy, const __nv_bfloat16* o, const int32_t* row_of,
                        const float* probs, int64_t T, int k, int H, __nv_bfloat16* d_o,
                        float* dprobs, cudaStream_t st);

// ------------------------------------------------------------------ MXFP8

// codes of x in permuted rows ([cap, H], uint8) and its scales in token
// order ([T, H/32], uint8).
cudaError_t launch_permute_quantize(const __nv_bfloat16* x, int64_t T, int H, int k,
                                    const int32_t* row_of, uint8_t* xq, uint8_t* xs_tok,
                                    cudaStream_t st, int64_t n_rows = -1, int* err = nullptr);
// token-order scales -> the tiled layout over the padded permuted rows.
cudaError_t launch_gather_tile_scales(const uint8_t* xs_tok, const int32_t* token_of,
                                      const int32_t* off_al, const int32_t* counts, int E, int K,
                                      int64_t cap, uint8_t* xs_tiled, cudaStream_t st);
// row-major scales -> tiled layout (see mx.cuh); pair_half > 0 interleaves
// the gate and up weights' rows per pair_half so that one N tile of
// 2*pair_half rows holds both halves.
cudaError_t launch_tile_scales(const uint8_t* src0, const uint8_t* src1, int64_t out_rows,
                               int64_t rows_per_e, int K, int pair_half, uint8_t* dst,
                               cudaStream_t st);

// Epilogues of the MXFP8 GEMMs: Fc1 = SwiGLU, h to bf16 and MXFP8 (codes +
// tiled scales), optionally saving A_g, A_u and h in bf16; Bf16 = rows of
// bf16 (fc2); SwigluBwd = dA_g, dA_u in bf16 from dH and the saved A_g, A_u;
// F32 = weight-gradient rows (WGrad schedule). Rows leave through the
// output tensor maps (make_out_tmap): fc2's O and dXp (bf16, map 0), the
// weight gradients (0, and 1 past out_split).
enum class MxEpi { Fc1, Bf16, SwigluBwd, F32, Fc1Save };   // Fc1Save: fc1 with p.save

struct MxGemmArgs {
  const int32_t* off_al;   // [E+1] padded expert row offsets
  int E;
  int K;                   // Rows: reduction length (elements = bytes)
  int N;                   // output columns (fc1: F, fc2: H, dH: F, dXp: H, WGrad: cols of B)
  int M;                   // WGrad: output rows per expert (rows of A)
  int stages;
  int bn;                  // MMA N: 128 or 256
  int64_t b_rows;          // Rows: rows of one expert in B's 2D view (fc1: F, fc2: H)
  int64_t sfb_rows;        // Rows: rows of one expert in B's tiled scales (fc1: 2F, fc2: H)
  int k_split;             // Rows: k-blocks taken from B0 before B1 (0: B0 only)
  int kgroups_a;           // 128-wide K groups in A's tiled scales (0: K / 128)
  int kgroups_b;           // 128-wide K groups in B's (and B1's) tiled scales (0: K / 128)
  int keep_a;              // L2 evict_last hint on A loads
  const uint8_t* sfa;      // tiled scales of A
  const uint8_t* sfb;      // tiled scales of B (B0)
  const uint8_t* sfb1;     // tiled scales of B1 (k_split)
  uint8_t* hq;             // fc1: codes of h [rows, N]
  uint8_t* hs;             // fc1: tiled scales of h
  int save;                // fc1: also store A_g, A_u and h in bf16, blocked
                           // (act_block_offset, N = F): save_g, save_u, save_h
  __nv_bfloat16* save_g;
  __nv_bfloat16* save_u;
  __nv_bfloat16* save_h;
  __nv_bfloat16* out_b;    // SwigluBwd: [dA_g | dA_u], blocked with N = 2 * N
  const __nv_bfloat16* act_g;   // SwigluBwd: saved A_g, A_u [rows, N], blocked
  const __nv_bfloat16* act_u;
  int out_split;           // WGrad: rows r < out_split of each expert go to output map 0
                           // (row e * out_split + r), the rest to map 1; 0 means M
  int accumulate;          // WGrad: add to the outputs instead of overwriting
  int pair;                // Rows: CTA pairs share M = 256 tiles
  int* err;
  unsigned long long wait_ns;
};

// Tensor maps over the tiled scale arrays (sfa, sfb, sfb1) as rows of 256
// bytes, one 512-byte atom per box of two rows (make_tmap_scale_rows): every
// MXFP8 GEMM loads its scale atoms through them (a tensor-map copy is cheap
// to issue; a CTA pair's copies can complete on the leader's barrier).
struct MxScaleMaps {
  CUtensorMap map[3];
};
bool make_tmap_scale_rows(CUtensorMap* map, const void* base, uint64_t bytes);
// The maps of one GEMM's scale arrays (sizes in bytes); without sfb1, map 2
// repeats map 1.
bool make_scale_maps(MxScaleMaps* m, const uint8_t* sfa, uint64_t sfa_bytes, const uint8_t* sfb,
                     uint64_t sfb_bytes, const uint8_t* sfb1 = nullptr, uint64_t sfb1_bytes = 0);

// The forward keeps A_g and A_u [rows, N] (rows, N % 32 == 0) in 32 x 32
// blocks of 2 KB, block (row / 32, col / 32) at ((row / 32) * (N / 32) +
// col / 32) * 1024 elements; inside a block, 8-column slab j of row r at
// j * 256 + r * 8. A warp that owns 32 rows then moves one 32-column chunk
// of them with four fully coalesced 512-byte accesses, lane r holding its
// own row (the TMEM lane layout of the accumulator).
__host__ __device__ __forceinline__ int64_t act_block_offset(int64_t row, int64_t col, int64_t N) {
  return ((row >> 5) * (N >> 5) + (col >> 5)) * 1024 + ((col & 31) >> 3) * 256 + (row & 31) * 8 +
         (col & 7);
}

// Encodes a 2D uint8 tensor map with the 128-byte swizzle.
bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

cudaError_t launch_mx_fc1(const CUtensorMap& a, const CUtensorMap& wg, const CUtensorMap& wu,
                          const GemmOut& o, const MxGemmArgs& p, int grid, cudaStream_t st,
                          const MxScaleMaps& sc);
// dH with the SwiGLU backward epilogue (Rows; B = W2 as [E*F, H] along H).
cudaError_t launch_mx_dh(const CUtensorMap& a, const CUtensorMap& w2, const GemmOut& o,
                         const MxGemmArgs& p, int grid, cudaStream_t st, const MxScaleMaps& sc);
// dXp = bf16(dA_g W1g^T + dA_u W1u^T) (Rows; K = 2F split over B0, B1).
cudaError_t launch_mx_dxp(const CUtensorMap& a, const CUtensorMap& w1g, const CUtensorMap& w1u,
                          const GemmOut& o, const MxGemmArgs& p, int grid, cudaStream_t st,
                          const MxScaleMaps& sc);
// Weight gradients (WGrad: K = each expert's padded rows), float out.
cudaError_t launch_mx_wgrad(const CUtensorMap& a, const CUtensorMap& b, const GemmOut& o,
                            const MxGemmArgs& p, int grid, cudaStream_t st, const MxScaleMaps& sc);
cudaError_t launch_mx_fc2(const CUtensorMap& a, const CUtensorMap& wd, const GemmOut& o,
                          const MxGemmArgs& p, int grid, cudaStream_t st, const MxScaleMaps& sc);

int device_sm_count();
// The current CUDA device, or -1; launchers keep per-device state indexed by
// it (kernel attributes are per device).
constexpr int kMaxDevices = 64;
int current_device();

}  // namespace moe
