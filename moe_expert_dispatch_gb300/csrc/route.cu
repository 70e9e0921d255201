// route.cu - the data-movement steps of the expert block: per-expert counts
// (histc), the offset scan, the stable row map, the permute gather, the
// probability-weighted unpermute and the MXFP8 quantiser. All are bound by
// HBM bandwidth (or latency, for the tiny count/scan kernels); rows move as
// 16-byte vectors, one warp per token so that each warp streams whole rows.
// They are the steps of ep_mc2_forward in "NPU Training Operators - MC2"
// (section "execution path") on one GPU: step 2 histc (hist_kernel), steps
// 4-5 (scan_kernel, send = receive = the local counts), step 6 permute
// (rowmap_kernel + permute_copy_kernel) and step 10 unpermute; the gate
// ahead of them is route_topk_kernel. The MXFP8 dispatch and quantisers
// follow the MX FP8 of "MC2 通算融合架构总览", section 1.
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "mx.cuh"

namespace moe {

// ------------------------------------------------------------------ counts

size_t route_scratch_bytes(int64_t n_ids, int E) {
  const int64_t c = route_chunks(n_ids > 0 ? n_ids : 1);
  const size_t one = static_cast<size_t>(c) * E * sizeof(int32_t);
  return kRouteHeadBytes + 2 * ((one + 255) / 256 * 256);
}

RouteScratch route_scratch(void* ws, int64_t n_ids, int E) {
  RouteScratch s;
  s.chunks = route_chunks(n_ids > 0 ? n_ids : 1);
  const size_t one = (static_cast<size_t>(s.chunks) * E * sizeof(int32_t) + 255) / 256 * 256;
  s.ticket = static_cast<unsigned int*>(ws);
  s.hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kRouteHeadBytes);
  s.base = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kRouteHeadBytes + one);
  return s;
}

// CTAs of warps_per_cta warps for one warp per work item, capped at 16 per SM
// (the kernels loop over the rest).
static int grid_for_warps(int64_t warps, int warps_per_cta) {
  const int64_t want = (warps + warps_per_cta - 1) / warps_per_cta;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

// One CTA per chunk of ids: a shared-memory histogram, with the lanes of a
// warp that hold the same expert folded into one atomic (match.any).
__global__ void __launch_bounds__(256) hist_kernel(const int32_t* __restrict__ ids, int64_t n,
                                                   int E, int32_t* __restrict__ hist, int* err) {
  extern __shared__ int sh_count[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh_count[e] = 0;
  __syncthreads();
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
  const int64_t hi = min(n, lo + kRouteChunk);
  bool bad = false;
  for (int64_t i0 = lo; i0 < hi; i0 += blockDim.x) {
    const int64_t i = i0 + threadIdx.x;
    int e = -1;
    if (i < hi) {
      e = __ldg(ids + i);
      if (e < 0 || e >= E) {
        bad = true;
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane_id() == __ffs(peers) - 1) atomicAdd(&sh_count[e], __popc(peers));
  }
  if (bad) report_error(err, kErrBadId);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    hist[static_cast<int64_t>(blockIdx.x) * E + e] = sh_count[e];
}

// Exclusive prefix sums of v[0..n) (n <= 1024) in place, by warp 0 of the
// CTA: lane l sums a segment of ceil(n / 32) entries, a warp scan offsets
// the segments, then each lane writes its segment's prefixes. The total goes
// to *total.
__device__ void warp0_exclusive_scan(int* v, int n, int* total) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int seg = (n + 31) >> 5;
  const int lo = min(n, lane * seg), hi = min(n, lo + seg);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += v[i];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  int run = incl - sum;
  for (int i = lo; i < hi; ++i) {
    const int x = v[i];
    v[i] = run;
    run += x;
  }
  if (lane == 31) *total = incl;
}

// Run by one CTA: per expert the total over the chunks, the dense and the
// padded offsets, then every chunk's first row (its padded expert offset
// plus the expert's ids in earlier chunks). hist is read through L2 (other
// CTAs of the same launch may have written it), with 8 loads in flight per
// expert, and is never read back after a write. Up to 32 experts one warp
// does it all in registers; beyond, warp 0 scans in shared memory.
__device__ void scan_chunks(const int32_t* hist, int32_t* base, int64_t chunks, int E, int align,
                            int32_t* counts, int32_t* offsets, int32_t* off_al, int* sh_cnt,
                            int* sh_al) {
  constexpr int U = 8;                     // independent loads in flight per expert
  constexpr int kRegChunks = 32;           // one pass from registers up to this many chunks
  __shared__ int total_dense, total_al;
  if (E <= 32) {
    // one warp, one expert per lane: totals, both scans by shuffles, bases
    if (threadIdx.x >= 32) return;
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
      for (int64_t c0 = 0; c0 < chunks; c0 += U) {
        int v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = c0 + u < chunks ? __ldcg(hist + (c0 + u) * E + e) : 0;
#pragma unroll
        for (int u = 0; u < U; ++u) run += v[u];
      }
    }
    const int al = (run + align - 1) / align * align;
    int inc = run, inc_al = al;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      const int ta = __shfl_up_sync(0xffffffffu, inc_al, o);
      if (e >= o) {
        inc += t;
        inc_al += ta;
      }
    }
    if (e < E) {
      if (counts) counts[e] = run;
      if (offsets) offsets[e] = inc - run;
      if (off_al) off_al[e] = inc_al - al;
    }
    if (e == 31) {
      if (offsets) offsets[E] = inc;
      if (off_al) off_al[E] = inc_al;
    }
    if (e < E) {
      int b = inc_al - al;
      for (int64_t c0 = 0; c0 < chunks; c0 += U) {
        int v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = c0 + u < chunks ? __ldcg(hist + (c0 + u) * E + e) : 0;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + u < chunks) {
            base[(c0 + u) * E + e] = b;
            b += v[u];
          }
      }
    }
    return;
  }
  // with one expert per thread and few chunks, the chunk values stay in
  // registers between the totals and the bases
  const bool one_pass = chunks <= kRegChunks && E <= static_cast<int>(blockDim.x);
  int keep[kRegChunks];
  if (one_pass) {
    const int e = threadIdx.x;
    if (e < E) {
      int run = 0;
#pragma unroll
      for (int u = 0; u < kRegChunks; ++u) {
        keep[u] = u < chunks ? __ldcg(hist + static_cast<int64_t>(u) * E + e) : 0;
        run += keep[u];
      }
      if (counts) counts[e] = run;
      sh_cnt[e] = run;
      sh_al[e] = (run + align - 1) / align * align;
    }
  } else {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int run = 0;
      for (int64_t c0 = 0; c0 < chunks; c0 += U) {
        int v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = c0 + u < chunks ? __ldcg(hist + (c0 + u) * E + e) : 0;
#pragma unroll
        for (int u = 0; u < U; ++u) run += v[u];
      }
      if (counts) counts[e] = run;
      sh_cnt[e] = run;
      sh_al[e] = (run + align - 1) / align * align;
    }
  }
  __syncthreads();
  warp0_exclusive_scan(sh_al, E, &total_al);
  if (offsets) warp0_exclusive_scan(sh_cnt, E, &total_dense);    // the same warp, in order
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    if (offsets) offsets[e] = sh_cnt[e];
    if (off_al) off_al[e] = sh_al[e];
  }
  if (threadIdx.x == 0) {
    if (offsets) offsets[E] = total_dense;
    if (off_al) off_al[E] = total_al;
  }
  if (one_pass) {
    const int e = threadIdx.x;
    if (e < E) {
      int run = sh_al[e];
#pragma unroll
      for (int u = 0; u < kRegChunks; ++u)
        if (u < chunks) {
          base[static_cast<int64_t>(u) * E + e] = run;
          run += keep[u];
        }
    }
    return;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = sh_al[e];
    for (int64_t c0 = 0; c0 < chunks; c0 += U) {
      int v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = c0 + u < chunks ? __ldcg(hist + (c0 + u) * E + e) : 0;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (c0 + u < chunks) {
          base[(c0 + u) * E + e] = run;
          run += v[u];
        }
    }
  }
}

__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ hist,
                                                    int32_t* __restrict__ base, int64_t chunks,
                                                    int E, int align, int32_t* counts,
                                                    int32_t* offsets, int32_t* off_al) {
  __shared__ int sh_cnt[kMaxExperts];
  __shared__ int sh_al[kMaxExperts];
  scan_chunks(hist, base, chunks, E, align, counts, offsets, off_al, sh_cnt, sh_al);
}

cudaError_t launch_counts(const int32_t* ids, int64_t n, int E, int align, int32_t* counts,
                          int32_t* offsets, int32_t* off_al, RouteScratch s, int* err,
                          cudaStream_t st) {
  const int64_t chunks = route_chunks(n);
  if (chunks > 0)
    hist_kernel<<<static_cast<unsigned>(chunks), 256, E * sizeof(int), st>>>(ids, n, E, s.hist,
                                                                            err);
  else
    cudaMemsetAsync(s.hist, 0, E * sizeof(int32_t), st);
  scan_kernel<<<1, 1024, 0, st>>>(s.hist, s.base, chunks > 0 ? chunks : 1, E, align, counts,
                                  offsets, off_al);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ gate (top-k + softmax + counts)

// Rank order of the gate: the larger logit first, equal logits (-0.0 and
// +0.0 included) to the lower expert index.
__device__ __forceinline__ bool ranks_before(float a, int ea, float b, int eb) {
  return a > b || (a == b && ea < eb);
}

// One warp per token. Lane l holds logits l, l + 32, ... (kEPL of them, NaN
// entered as -inf); k rounds of a warp arg-max in rank order pick the
// experts, lane j keeping the j-th pick. The weights are a float softmax
// over the chosen k. Every slot adds one to the histogram row of its
// 2048-id chunk (global atomics on rows cleared before the launch), so the
// row map and its chunk bases work as after launch_counts; the CTA that
// takes the last ticket runs the offset scan.
template <int kEPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits,
                                                         int64_t T, int E, int k, int align,
                                                         int32_t* __restrict__ ids,
                                                         float* __restrict__ probs, RouteScratch s,
                                                         int32_t* counts, int32_t* offsets,
                                                         int32_t* off_al) {
  __shared__ int sh_cnt[kMaxExperts];
  __shared__ int sh_al[kMaxExperts];
  __shared__ int is_last;
  const int lane = lane_id();
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       t < T; t += warps) {
    const float* row = logits + t * E;
    float v[kEPL];
    unsigned open = 0;                               // bit i: logit lane + 32 i not yet taken
#pragma unroll
    for (int i = 0; i < kEPL; ++i) {
      const int e = lane + 32 * i;
      float x = -INFINITY;
      if (e < E) {
        x = __ldg(row + e);
        if (isnan(x)) x = -INFINITY;
        open |= 1u << i;
      }
      v[i] = x;
    }
    float mine_v = 0.0f;
    int mine_e = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = INT_MAX;                              // ranks after every real expert
#pragma unroll
      for (int i = 0; i < kEPL; ++i)
        if (((open >> i) & 1u) && ranks_before(v[i], lane + 32 * i, bv, be)) {
          bv = v[i];
          be = lane + 32 * i;
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ranks_before(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      // k <= E, so every round finds an open expert: 0 <= be < E
      if ((be & 31) == lane) open &= ~(1u << (be >> 5));
      if (lane == j) {
        mine_v = bv;
        mine_e = be;
      }
    }
    const float top = __shfl_sync(0xffffffffu, mine_v, 0);
    const float ex = lane < k ? expf(mine_v - top) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) {
      const int64_t i = t * k + lane;
      ids[i] = mine_e;
      probs[i] = ex / sum;
      atomicAdd(s.hist + (i / kRouteChunk) * E + mine_e, 1);
    }
  }
  // the last CTA to finish sees every histogram row
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(s.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  scan_chunks(s.hist, s.base, s.chunks, E, align, counts, offsets, off_al, sh_cnt, sh_al);
  if (threadIdx.x == 0) *s.ticket = 0;
}

template <int kEPL>
static void launch_route_topk_epl(const float* logits, int64_t T, int E, int k, int align,
                                  int32_t* ids, float* probs, RouteScratch s, int32_t* counts,
                                  int32_t* offsets, int32_t* off_al, cudaStream_t st) {
  route_topk_kernel<kEPL><<<grid_for_warps(T, 8), 256, 0, st>>>(logits, T, E, k, align, ids, probs,
                                                                s, counts, offsets, off_al);
}

cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int align,
                              int32_t* ids, float* probs, int32_t* counts, int32_t* offsets,
                              int32_t* off_al, RouteScratch s, cudaStream_t st) {
  const size_t hist_bytes = static_cast<size_t>(s.chunks) * E * sizeof(int32_t);
  cudaError_t e = cudaMemsetAsync(s.ticket, 0, kRouteHeadBytes + hist_bytes, st);
  if (e != cudaSuccess) return e;
  if (E <= 32)
    launch_route_topk_epl<1>(logits, T, E, k, align, ids, probs, s, counts, offsets, off_al, st);
  else if (E <= 64)
    launch_route_topk_epl<2>(logits, T, E, k, align, ids, probs, s, counts, offsets, off_al, st);
  else if (E <= 128)
    launch_route_topk_epl<4>(logits, T, E, k, align, ids, probs, s, counts, offsets, off_al, st);
  else if (E <= 256)
    launch_route_topk_epl<8>(logits, T, E, k, align, ids, probs, s, counts, offsets, off_al, st);
  else if (E <= 512)
    launch_route_topk_epl<16>(logits, T, E, k, align, ids, probs, s, counts, offsets, off_al, st);
  else
    launch_route_topk_epl<32>(logits, T, E, k, align, ids, probs, s, counts, offsets, off_al, st);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ row map

// One CTA per chunk; warp w owns 256 consecutive ids, taken 32 at a time, so
// the order "chunk, warp, step, lane" is the flat-index order. Pass 1 counts
// per (warp, expert); a scan over warps turns that into each warp's first
// row; pass 2 gives every id its row = warp base + rank among equal lanes.
constexpr int kRowmapWarps = 8;
constexpr int kRowmapPerWarp = kRouteChunk / kRowmapWarps;

__global__ void __launch_bounds__(256) rowmap_kernel(const int32_t* __restrict__ ids,
                                                     const float* __restrict__ probs, int64_t n,
                                                     int k, int E,
                                                     const int32_t* __restrict__ base,
                                                     int32_t* __restrict__ row_of,
                                                     int32_t* __restrict__ token_of,
                                                     float* __restrict__ prob_of,
                                                     int64_t n_rows, int* err) {
  extern __shared__ int wc[];  // [kRowmapWarps][E]
  for (int i = threadIdx.x; i < kRowmapWarps * E; i += blockDim.x) wc[i] = 0;
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = lane_id();
  const int64_t start = static_cast<int64_t>(blockIdx.x) * kRouteChunk + w * kRowmapPerWarp;
  const unsigned lt = (1u << lane) - 1u;
  for (int s = 0; s < kRowmapPerWarp; s += 32) {
    const int64_t i = start + s + lane;
    int e = (i < n) ? __ldg(ids + i) : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wc[w * E + e] += __popc(peers);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = base[static_cast<int64_t>(blockIdx.x) * E + e];
    for (int q = 0; q < kRowmapWarps; ++q) {
      const int v = wc[q * E + e];
      wc[q * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  for (int s = 0; s < kRowmapPerWarp; s += 32) {
    const int64_t i = start + s + lane;
    int e = (i < n) ? __ldg(ids + i) : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int r = -1;
    if (e >= 0) r = wc[w * E + e] + __popc(peers & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wc[w * E + e] += __popc(peers);
    __syncwarp();
    if (i < n) {
      row_of[i] = r;
      if (r >= 0 && dbg_row_ok(r, n_rows, err)) {
        token_of[r] = static_cast<int32_t>(i / k);
        if (prob_of) prob_of[r] = probs ? __ldg(probs + i) : 1.0f;
      }
    }
  }
}

cudaError_t launch_rowmap(const int32_t* ids, const float* probs, int64_t n, int k, int E,
                          RouteScratch s, int32_t* row_of, int32_t* token_of, float* prob_of,
                          cudaStream_t st, int64_t n_rows, int* err) {
  const int64_t chunks = route_chunks(n);
  if (chunks == 0) return cudaSuccess;
  rowmap_kernel<<<static_cast<unsigned>(chunks), 256, kRowmapWarps * E * sizeof(int), st>>>(
      ids, probs, n, k, E, s.base, row_of, token_of, prob_of, n_rows, err);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ permute copy

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// One warp per token: the token's row is read once and written to its k
// rows; each warp instruction moves 512 contiguous bytes.
__global__ void __launch_bounds__(256) permute_copy_kernel(const uint8_t* __restrict__ x,
                                                           int64_t T, int64_t row_bytes, int k,
                                                           const int32_t* __restrict__ row_of,
                                                           uint8_t* __restrict__ xp,
                                                           int64_t n_rows, int* err) {
  constexpr int U = 4;
  const int lane = lane_id();
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t n16 = row_bytes >> 4;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       t < T; t += warps) {
    const int my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
    const int4* src = reinterpret_cast<const int4*>(x + t * row_bytes);
    // the trip count is the same for every lane (the shuffles below need the
    // whole warp); lanes past the row end just skip their vectors
    for (int64_t base = 0; base < n16; base += 32 * U) {
      const int64_t c0 = base + lane;
      int4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (c0 + 32 * u < n16) v[u] = ld_stream(src + c0 + 32 * u);
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_row, j);
        if (r < 0 || !dbg_row_ok(r, n_rows, err)) continue;   // warp-uniform
        int4* dst = reinterpret_cast<int4*>(xp + static_cast<int64_t>(r) * row_bytes);
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + 32 * u < n16) dst[c0 + 32 * u] = v[u];
      }
    }
  }
}

cudaError_t launch_permute_copy(const void* x, int64_t T, int64_t row_bytes, int k,
                                const int32_t* row_of, void* xp, cudaStream_t st, int64_t n_rows,
                                int* err) {
  if (T == 0) return cudaSuccess;
  permute_copy_kernel<<<grid_for_warps(T, 8), 256, 0, st>>>(
      static_cast<const uint8_t*>(x), T, row_bytes, k, row_of, static_cast<uint8_t*>(xp), n_rows,
      err);
  return cudaGetLastError();
}

// blockIdx.y = expert; the CTA zeroes rows [off_al[e] + c_e, off_al[e+1]).
__global__ void __launch_bounds__(256) zero_padding_kernel(const int32_t* __restrict__ counts,
                                                           const int32_t* __restrict__ off_al,
                                                           int64_t row_bytes, uint8_t* xp,
                                                           int32_t* token_of, float* prob_of) {
  const int e = blockIdx.y;
  const int64_t r0 = off_al[e] + counts[e], r1 = off_al[e + 1];
  const int64_t n16 = (r1 - r0) * (row_bytes >> 4);
  int4* base = reinterpret_cast<int4*>(xp + r0 * row_bytes);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    base[i] = make_int4(0, 0, 0, 0);
  if (blockIdx.x == 0)
    for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
      if (token_of) token_of[r] = -1;
      if (prob_of) prob_of[r] = 0.0f;
    }
}

cudaError_t launch_zero_padding(const int32_t* counts, const int32_t* off_al, int E,
                                int64_t row_bytes, void* xp, int32_t* token_of, float* prob_of,
                                cudaStream_t st) {
  const int64_t per = static_cast<int64_t>(kTileM - 1) * (row_bytes >> 4);
  const int gx = static_cast<int>((per + 255) / 256 < 64 ? (per + 255) / 256 : 64);
  zero_padding_kernel<<<dim3(gx > 0 ? gx : 1, E), 256, 0, st>>>(
      counts, off_al, row_bytes, static_cast<uint8_t*>(xp), token_of, prob_of);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ unpermute

__device__ __forceinline__ void acc_bf16x8(float* acc, const int4& v, float p) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(h[q]);
    acc[2 * q] = fmaf(p, f.x, acc[2 * q]);
    acc[2 * q + 1] = fmaf(p, f.y, acc[2 * q + 1]);
  }
}

// y[t] = bf16(sum_j p_j o[row_j]), j in order, float accumulation. One warp
// per (token, column chunk of 32 lanes x kUnpermU 16-byte vectors): a short
// row count still gives every SM a full set of warps. Slot pairs are loaded
// together so two rows are in flight before either is accumulated.
constexpr int kUnpermU = 2;

__global__ void __launch_bounds__(256) unpermute_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const int32_t* __restrict__ row_of,
                                                        const float* __restrict__ probs,
                                                        int64_t T, int k, int H,
                                                        __nv_bfloat16* __restrict__ y,
                                                        int64_t n_rows, int* err) {
  constexpr int U = kUnpermU;
  const int lane = lane_id();
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int n8 = H >> 3;
  const int chunks = (n8 + 32 * U - 1) / (32 * U);
  const int64_t tasks = T * chunks;
  for (int64_t task = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       task < tasks; task += warps) {
    const int64_t t = task / chunks;
    const int c0 = static_cast<int>(task - t * chunks) * 32 * U + lane;
    const int my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
    const float my_p = lane < k ? (probs ? __ldg(probs + t * k + lane) : 1.0f) : 0.0f;
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[u][q] = 0.0f;
    for (int j = 0; j < k; j += 2) {            // warp-uniform trip count
      int r0 = __shfl_sync(0xffffffffu, my_row, j);
      const float p0 = __shfl_sync(0xffffffffu, my_p, j);
      int r1 = __shfl_sync(0xffffffffu, my_row, (j + 1) & 31);
      if (r0 >= 0 && !dbg_row_ok(r0, n_rows, err)) r0 = -1;      // warp-uniform
      if (r1 >= 0 && !dbg_row_ok(r1, n_rows, err)) r1 = -1;
      const float p1 = __shfl_sync(0xffffffffu, my_p, (j + 1) & 31);
      const bool has1 = j + 1 < k && r1 >= 0;
      int4 v0[U], v1[U];
      if (r0 >= 0) {
        const int4* src = reinterpret_cast<const int4*>(o + static_cast<int64_t>(r0) * H);
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + 32 * u < n8) v0[u] = ld_stream(src + c0 + 32 * u);
      }
      if (has1) {
        const int4* src = reinterpret_cast<const int4*>(o + static_cast<int64_t>(r1) * H);
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + 32 * u < n8) v1[u] = ld_stream(src + c0 + 32 * u);
      }
      if (r0 >= 0) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + 32 * u < n8) acc_bf16x8(acc[u], v0[u], p0);
      }
      if (has1) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + 32 * u < n8) acc_bf16x8(acc[u], v1[u], p1);
      }
    }
    int4* dst = reinterpret_cast<int4*>(y + t * H);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c0 + 32 * u < n8) {
        int4 w;
        w.x = static_cast<int>(pack_bf16x2(acc[u][0], acc[u][1]));
        w.y = static_cast<int>(pack_bf16x2(acc[u][2], acc[u][3]));
        w.z = static_cast<int>(pack_bf16x2(acc[u][4], acc[u][5]));
        w.w = static_cast<int>(pack_bf16x2(acc[u][6], acc[u][7]));
        dst[c0 + 32 * u] = w;
      }
  }
}

cudaError_t launch_unpermute(const __nv_bfloat16* o, const int32_t* row_of, const float* probs,
                             int64_t T, int k, int H, __nv_bfloat16* y, cudaStream_t st,
                             int64_t n_rows, int* err) {
  if (T == 0) return cudaSuccess;
  const int64_t chunks = ((H >> 3) + 32 * kUnpermU - 1) / (32 * kUnpermU);
  unpermute_kernel<<<grid_for_warps(T * chunks, 8), 256, 0, st>>>(o, row_of, probs, T, k, H, y,
                                                                  n_rows, err);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ backward: dO, dprobs

// One warp per token t: for each of its slots j (8 at a time) the warp
// streams dY_t once and O[row_j]: dO[row_j] = bf16(p_tj dY_t) and
// dprobs[t, j] = <dY_t, O[row_j]> (float, reduced across the warp).
__global__ void __launch_bounds__(256) dout_kernel(const __nv_bfloat16* __restrict__ dy,
                                                   const __nv_bfloat16* __restrict__ o,
                                                   const int32_t* __restrict__ row_of,
                                                   const float* __restrict__ probs, int64_t T,
                                                   int k, int H, __nv_bfloat16* __restrict__ d_o,
                                                   float* __restrict__ dprobs) {
  const int lane = lane_id();
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int n8 = H >> 3;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       t < T; t += warps) {
    const int my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
    const float my_p = lane < k ? __ldg(probs + t * k + lane) : 0.0f;
    const int4* g4 = reinterpret_cast<const int4*>(dy + t * H);
    for (int j0 = 0; j0 < k; j0 += 8) {
      float dot[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) dot[q] = 0.0f;
      for (int base = 0; base < n8; base += 32) {   // warp-uniform trip count
        const int c = base + lane;
        float gf[8];
        if (c < n8) {
          const int4 g = ld_stream(g4 + c);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(h[q]);
            gf[2 * q] = f.x;
            gf[2 * q + 1] = f.y;
          }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          if (j >= k) break;
          const int r = __shfl_sync(0xffffffffu, my_row, j);
          const float p = __shfl_sync(0xffffffffu, my_p, j);
          if (r < 0 || c >= n8) continue;
          const int4 ov = ld_stream(reinterpret_cast<const int4*>(o + static_cast<int64_t>(r) * H) + c);
          const __nv_bfloat162* oh = reinterpret_cast<const __nv_bfloat162*>(&ov);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(oh[q]);
            dot[jj] = fmaf(gf[2 * q], f.x, dot[jj]);
            dot[jj] = fmaf(gf[2 * q + 1], f.y, dot[jj]);
          }
          int4 w;
          w.x = static_cast<int>(pack_bf16x2(p * gf[0], p * gf[1]));
          w.y = static_cast<int>(pack_bf16x2(p * gf[2], p * gf[3]));
          w.z = static_cast<int>(pack_bf16x2(p * gf[4], p * gf[5]));
          w.w = static_cast<int>(pack_bf16x2(p * gf[6], p * gf[7]));
          reinterpret_cast<int4*>(d_o + static_cast<int64_t>(r) * H)[c] = w;
        }
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        float v = dot[jj];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        const int j = j0 + jj;
        if (lane == 0 && j < k) dprobs[t * k + j] = v;
      }
    }
  }
}

cudaError_t launch_dout(const __nv_bfloat16* dy, const __nv_bfloat16* o, const int32_t* row_of,
                        const float* probs, int64_t T, int k, int H, __nv_bfloat16* d_o,
                        float* dprobs, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  dout_kernel<<<grid_for_warps(T, 8), 256, 0, st>>>(dy, o, row_of, probs, T, k, H, d_o, dprobs);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ MXFP8

// Quantisation along the rows: four lanes per 32-element block, each with 8
// consecutive elements (one 16-byte load, one 8-byte store), so a warp reads
// 512 and writes 256 contiguous bytes per block group, with four such loads
// in flight per lane; the block's amax is a max over the four lanes. Scales row-major [rows, K/32], or (kTiled) in the tiled layout
// of the block-scaled MMA (rows % 128 == 0, K % 128 == 0); with row_end,
// rows at or past *row_end are skipped (the unused tail of a padded layout).
template <bool kTiled>
__global__ void __launch_bounds__(256) quantize_mxfp8_kernel(const __nv_bfloat16* __restrict__ in,
                                                             int64_t blocks, int K,
                                                             const int32_t* __restrict__ row_end,
                                                             uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ scales) {
  constexpr int kU = 4;                    // items per lane per pass, loaded together
  const int nb = K >> 5;
  const int64_t limit = row_end ? static_cast<int64_t>(*row_end) * nb : blocks;
  const int64_t end = 4 * (limit < blocks ? limit : blocks);     // (block, quarter) items
  const int lane = lane_id();
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  // warp-uniform trip count: the shuffles below need every lane. A pass of
  // a warp covers kU consecutive runs of 32 items.
  for (int64_t base = (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) *
                      (32 * kU);
       base < end; base += warps * 32 * kU) {
    int4 raw[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t item = base + 32 * u + lane;
      raw[u] = item < end ? ld_stream(reinterpret_cast<const int4*>(in + (item >> 2) * 32 +
                                                                    (lane & 3) * 8))
                          : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t item = base + 32 * u + lane;
      const int64_t b = item >> 2;
      const int part = lane & 3;
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
      float v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        v[2 * j] = f.x;
        v[2 * j + 1] = f.y;
      }
      uint32_t amax = bf16x2_absmax_bits<4>(reinterpret_cast<const uint32_t*>(&raw[u]));
      amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int code = mx_block_code(amax);
      const float inv = mx_inv_scale(code);
      if (item < end) {
        uint2 w;
        w.x = mx_encode4(v[0], v[1], v[2], v[3], inv);
        w.y = mx_encode4(v[4], v[5], v[6], v[7], inv);
        if (code == kMxNanScale) w = make_uint2(kMxNanCodes, kMxNanCodes);
        *reinterpret_cast<uint2*>(q + b * 32 + part * 8) = w;
        if (part == 0) {
          const uint8_t sc = static_cast<uint8_t>(code);
          if (kTiled)
            scales[mx_scale_offset(b / nb, b % nb, K)] = sc;
          else
            scales[b] = sc;
        }
      }
    }
  }
}

static unsigned grid_for_blocks(int64_t blocks) {
  const int64_t want = (blocks + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  return static_cast<unsigned>(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_quantize_mxfp8(const __nv_bfloat16* in, int64_t rows, int K, uint8_t* q,
                                  uint8_t* scales, cudaStream_t st) {
  const int64_t blocks = rows * (K / 32);
  if (blocks == 0) return cudaSuccess;
  quantize_mxfp8_kernel<false><<<grid_for_blocks(blocks), 256, 0, st>>>(in, blocks, K, nullptr, q,
                                                                        scales);
  return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp8_tiled(const __nv_bfloat16* in, int64_t rows, int K,
                                        const int32_t* row_end, uint8_t* q, uint8_t* scales,
                                        cudaStream_t st) {
  const int64_t blocks = rows * (K / 32);
  if (blocks == 0) return cudaSuccess;
  quantize_mxfp8_kernel<true><<<grid_for_blocks(blocks), 256, 0, st>>>(in, blocks, K, row_end, q,
                                                                       scales);
  return cudaGetLastError();
}

// Quantisation along the rows (the transposed orientation), alone or with
// the row orientation from the same read. For each batch z and column c of
// in[z] [rows, cols], the 32-row blocks of that column become 32
// K-contiguous codes of q_col[z] [cols, rows] and one scale, row-major
// [z, cols, rows/32] or (kTiled) tiled for an operand of batch * cols rows
// and K = rows. With kDual, the rows' 32-column blocks also become q_row
// [batch * rows, cols] with scales row-major [batch * rows, cols/32] or tiled
// (K = cols), by the rule of quantize_mxfp8_kernel.
//
// A CTA of 256 threads takes a tile of 128 rows x 128 columns. Its loads
// are coalesced 256-byte row pieces, all eight of a thread in flight at
// once, staged in shared memory in swizzled 16-byte chunks so that every
// access pattern below is free of bank conflicts. Along the
// rows (kDual) each lane quantises a whole 32-column block (one scale per
// lane, no shuffles) and writes its 32 codes. Down the columns, each thread
// quantises two 32-row blocks of one column; the codes gather in shared
// memory, a column's 128 codes in one 128-byte row, and leave as whole
// lines, so that the column codes, which land 32 bytes per output row per
// row block, reach L2 as full-line writes. With gather, row r of in is
// in[gather[r]] (a routed row of x), and a row whose gather index is outside
// [0, src_rows) is zero (padding). With row_end, rows at or past *row_end
// are skipped in whole 32-row blocks; the rest of a live block is zero.
// rows % 32 == 0; cols % 8 == 0 (kDual: cols % 128 == 0); kTiled: rows and
// cols % 128 == 0.
constexpr int kQtRows = 128, kQtCols = 128, kQtThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 16-byte chunk j of staged row r sits at chunk j ^ qt_swizzle(r): eight
// consecutive rows, or rows 64 apart, never share a bank group
__device__ __forceinline__ int qt_swizzle(int r) { return (r & 7) ^ ((r >> 4) & 4); }


// Where the bf16 input comes from: rows of a row-major matrix, gathered
// rows, or the 32 x 32 blocked layout of act_block_offset (with N = cols).
enum class QtSrc { Rows, Gather, Blocked };

template <bool kTiled, bool kDual, QtSrc kSrc>
__global__ void __launch_bounds__(kQtThreads) quantize_tile_kernel(
    const __nv_bfloat16* __restrict__ in, int64_t ld, int64_t batch_stride, int rows, int cols,
    const int32_t* __restrict__ gather, int64_t src_rows, const int32_t* __restrict__ row_end,
    uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row, uint8_t* __restrict__ q_col,
    uint8_t* __restrict__ s_col) {
  // 48 KB in all, so that four CTAs share an SM
  __shared__ __align__(16) uint8_t tile[kQtRows][kQtCols * 2];     // bf16, chunk-swizzled
  __shared__ __align__(16) uint8_t codes[kQtCols][kQtRows];        // column codes, swizzled
  const int r0 = blockIdx.x * kQtRows, c0 = blockIdx.y * kQtCols, z = blockIdx.z;
  const int live_rows = min(kQtRows, (row_end ? min(rows, *row_end) : rows) - r0);
  if (live_rows <= 0) return;
  const int n_rb = (live_rows + 31) >> 5;
  const __nv_bfloat16* base = in + static_cast<int64_t>(z) * batch_stride;
  const int tid = threadIdx.x;
  // load i of this thread: tile row lr(i), 8-column chunk ch(i). Row-major
  // sources: 16 lanes per 256-byte row piece. Blocked: a warp load is one
  // 512-byte slab (8 columns of a block's 32 rows, lane = row); the tile's
  // 16 blocks x 4 slabs are the 8 warps' 8 loads.
  auto load_row = [&](int i) {
    return kSrc == QtSrc::Blocked ? (((tid >> 5) * 8 + i) >> 4) * 32 + (tid & 31)
                                  : (tid >> 4) + 16 * i;
  };
  auto load_chunk = [&](int i) {
    const int q = (tid >> 5) * 8 + i;
    return kSrc == QtSrc::Blocked ? ((q >> 2) & 3) * 4 + (q & 3) : (tid & 15);
  };
  int4 v4[kQtRows / 16];
#pragma unroll
  for (int i = 0; i < kQtRows / 16; ++i) {
    const int lr = load_row(i), ch = load_chunk(i);
    int64_t r = r0 + lr;
    bool ok = lr < live_rows && c0 + ch * 8 < cols;
    if (kSrc == QtSrc::Gather && ok) {
      r = __ldg(gather + r);
      ok = r >= 0 && r < src_rows;
    }
    const __nv_bfloat16* src = kSrc == QtSrc::Blocked ? base + act_block_offset(r, c0 + ch * 8, cols)
                                                       : base + r * ld + c0 + ch * 8;
    v4[i] = ok ? ld_stream(reinterpret_cast<const int4*>(src)) : make_int4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kQtRows / 16; ++i) {
    const int lr = load_row(i), ch = load_chunk(i);
    *reinterpret_cast<int4*>(&tile[lr][(ch ^ qt_swizzle(lr)) << 4]) = v4[i];
  }
  __syncthreads();
  if (kDual) {
#pragma unroll 1
    for (int k = 0; k < 2; ++k) {
      const int r = (tid >> 2) + 64 * k, b = tid & 3;     // row, 32-column block
      if (r >= live_rows) break;
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 q = *reinterpret_cast<const uint4*>(&tile[r][((4 * b + j) ^ qt_swizzle(r)) << 4]);
        w[4 * j] = q.x;
        w[4 * j + 1] = q.y;
        w[4 * j + 2] = q.z;
        w[4 * j + 3] = q.w;
      }
      const int code = mx_block_code(bf16x2_absmax_bits<16>(w));
      const float inv = mx_inv_scale(code);
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        o[j] = mx_encode4(bf16_lo(w[2 * j]), bf16_hi(w[2 * j]), bf16_lo(w[2 * j + 1]),
                          bf16_hi(w[2 * j + 1]), inv);
        if (code == kMxNanScale) o[j] = kMxNanCodes;
      }
      const int64_t grow = static_cast<int64_t>(z) * rows + r0 + r;
      int4* dst = reinterpret_cast<int4*>(q_row + grow * cols + c0 + b * 32);
      dst[0] = make_int4(o[0], o[1], o[2], o[3]);
      dst[1] = make_int4(o[4], o[5], o[6], o[7]);
      const int kb = (c0 >> 5) + b;
      const uint8_t sc = static_cast<uint8_t>(code);
      if (kTiled)
        s_row[mx_scale_offset(grow, kb, cols)] = sc;
      else
        s_row[grow * (cols >> 5) + kb] = sc;
    }
  }
  // columns: lane l of warp w takes column c = 16 w + (l & 15) and its row
  // blocks 2p, 2p + 1, p = l >> 4, so that a column's four scales meet in one
  // warp (the swizzle keeps the halves, 64 rows apart, on disjoint banks).
  const int lane = tid & 31;
  const int c = 16 * (tid >> 5) + (lane & 15), p = lane >> 4;
  const bool col_ok = c0 + c < cols;
  uint32_t sc2 = 0;
  if (col_ok) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rb = 2 * p + h;
      if (rb < n_rb) {
        float v[32];
        uint32_t v2[16];                     // the same values as bf16 pairs
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int rr = rb * 32 + i;
          const uint32_t lo = *reinterpret_cast<const uint16_t*>(
              &tile[rr][(((c >> 3) ^ qt_swizzle(rr)) << 4) + (c & 7) * 2]);
          const uint32_t hi = *reinterpret_cast<const uint16_t*>(
              &tile[rr + 1][(((c >> 3) ^ qt_swizzle(rr + 1)) << 4) + (c & 7) * 2]);
          v2[i / 2] = lo | (hi << 16);
          v[i] = __uint_as_float(lo << 16);
          v[i + 1] = __uint_as_float(hi << 16);
        }
        const int code = mx_block_code(bf16x2_absmax_bits<16>(v2));
        const float inv = mx_inv_scale(code);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[i] = mx_encode4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], inv);
          if (code == kMxNanScale) w[i] = kMxNanCodes;
        }
        *reinterpret_cast<int4*>(&codes[c][((2 * rb) ^ (c & 7)) << 4]) =
            make_int4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<int4*>(&codes[c][((2 * rb + 1) ^ (c & 7)) << 4]) =
            make_int4(w[4], w[5], w[6], w[7]);
        sc2 |= static_cast<uint32_t>(code) << (8 * h);
      }
    }
  }
  // the column's n_rb (<= 4) scales are adjacent bytes in both layouts
  // (tiled: the 32-blocks kk = 0..3 of one 128-row K group); lane l < 16
  // writes them, one word when it can
  sc2 |= __shfl_xor_sync(0xffffffffu, sc2, 16) << 16;
  if (p == 0 && col_ok) {
    const int64_t orow = static_cast<int64_t>(z) * cols + c0 + c;
    const int64_t kb0 = r0 >> 5;
    uint8_t* d = kTiled ? s_col + mx_scale_offset(orow, kb0, rows) : s_col + orow * (rows >> 5) + kb0;
    if (n_rb == 4 && (reinterpret_cast<uintptr_t>(d) & 3) == 0) {
      *reinterpret_cast<uint32_t*>(d) = sc2;
    } else {
      for (int rb = 0; rb < n_rb; ++rb) d[rb] = static_cast<uint8_t>(sc2 >> (8 * rb));
    }
  }
  __syncthreads();
  // the column codes leave as whole rows of q_col: 8 lanes per 128-byte line
#pragma unroll
  for (int k = 0; k < (kQtCols * kQtRows / 16) / kQtThreads; ++k) {
    const int e = tid + kQtThreads * k;
    const int row = e >> 3, cc = e & 7;
    if ((cc >> 1) < n_rb && c0 + row < cols) {
      const int4 val = *reinterpret_cast<const int4*>(&codes[row][(cc ^ (row & 7)) << 4]);
      *reinterpret_cast<int4*>(q_col + (static_cast<int64_t>(z) * cols + c0 + row) * rows + r0 +
                               cc * 16) = val;
    }
  }
}

template <bool kDual>
static cudaError_t launch_quantize_tiles(const __nv_bfloat16* in, int64_t ld, int64_t batch,
                                         int64_t batch_stride, int rows, int cols,
                                         const int32_t* gather, int64_t src_rows,
                                         const int32_t* row_end, bool tiled, bool blocked,
                                         uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                                         uint8_t* s_col, cudaStream_t st) {
  if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((rows + kQtRows - 1) / kQtRows),
                  static_cast<unsigned>((cols + kQtCols - 1) / kQtCols),
                  static_cast<unsigned>(batch));
  auto kern = blocked  ? (tiled ? quantize_tile_kernel<true, kDual, QtSrc::Blocked>
                                : quantize_tile_kernel<false, kDual, QtSrc::Blocked>)
              : gather ? (tiled ? quantize_tile_kernel<true, kDual, QtSrc::Gather>
                                : quantize_tile_kernel<false, kDual, QtSrc::Gather>)
                       : (tiled ? quantize_tile_kernel<true, kDual, QtSrc::Rows>
                                : quantize_tile_kernel<false, kDual, QtSrc::Rows>);
  kern<<<grid, kQtThreads, 0, st>>>(in, ld, batch_stride, rows, cols, gather, src_rows, row_end,
                                    q_row, s_row, q_col, s_col);
  return cudaGetLastError();
}

cudaError_t launch_quantize_dual(const __nv_bfloat16* in, int64_t ld, int64_t batch,
                                 int64_t batch_stride, int rows, int cols,
                                 const int32_t* row_end, bool tiled, uint8_t* q_row,
                                 uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                 cudaStream_t st) {
  return launch_quantize_tiles<true>(in, ld, batch, batch_stride, rows, cols, nullptr, 0, row_end,
                                     tiled, false, q_row, s_row, q_col, s_col, st);
}

cudaError_t launch_quantize_dual_blocked(const __nv_bfloat16* in, int rows, int cols,
                                         const int32_t* row_end, uint8_t* q_row, uint8_t* s_row,
                                         uint8_t* q_col, uint8_t* s_col, cudaStream_t st) {
  return launch_quantize_tiles<true>(in, cols, 1, 0, rows, cols, nullptr, 0, row_end, true, true,
                                     q_row, s_row, q_col, s_col, st);
}

cudaError_t launch_quantize_cols(const __nv_bfloat16* in, int64_t ld, int64_t batch,
                                 int64_t batch_stride, int rows, int cols, const int32_t* gather,
                                 int64_t src_rows, const int32_t* row_end, bool tiled, uint8_t* q,
                                 uint8_t* scales, cudaStream_t st) {
  return launch_quantize_tiles<false>(in, ld, batch, batch_stride, rows, cols, gather, src_rows,
                                      row_end, tiled, false, nullptr, nullptr, q, scales, st);
}

cudaError_t launch_quantize_cols_blocked(const __nv_bfloat16* in, int rows, int cols,
                                         const int32_t* row_end, uint8_t* q, uint8_t* scales,
                                         cudaStream_t st) {
  return launch_quantize_tiles<false>(in, cols, 1, 0, rows, cols, nullptr, 0, row_end, true, true,
                                      nullptr, nullptr, q, scales, st);
}

// The dispatch of the MXFP8 path: one warp per token reads the bf16 row once,
// quantises it per 32 (the rule of quantize_mxfp8_kernel), writes the codes
// to each of the token's k rows and the scales once, in token order
// (row-major [T, H/32]); gather_tile_scales_kernel then lays the scales out
// per permuted row in the tiled layout. As in quantize_mxfp8_kernel, four
// lanes share a 32-element block, 8 consecutive elements each, so every warp
// load reads 512 contiguous bytes and every store to a row writes 256; a
// pass covers 32 blocks with four loads in flight per lane.
__global__ void __launch_bounds__(256) permute_quantize_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t T, int H, int k,
    const int32_t* __restrict__ row_of, uint8_t* __restrict__ xq, uint8_t* __restrict__ xs_tok,
    int64_t n_rows, int* err) {
  constexpr int kU = 4;                      // groups of 8 blocks per pass
  const int lane = lane_id();
  const int part = lane & 3;                 // which 8 elements of the block
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int nb = H >> 5;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       t < T; t += warps) {
    const int my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
    const __nv_bfloat16* src = x + t * H;
    for (int base = 0; base < nb; base += 8 * kU) {   // warp-uniform trip count
      int4 raw[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int b = base + 8 * u + (lane >> 2);
        raw[u] = b < nb ? ld_stream(reinterpret_cast<const int4*>(src + b * 32 + part * 8))
                        : make_int4(0, 0, 0, 0);
      }
      uint2 w[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int b = base + 8 * u + (lane >> 2);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
        float v[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(h[j]);
          v[2 * j] = f.x;
          v[2 * j + 1] = f.y;
        }
        uint32_t amax = bf16x2_absmax_bits<4>(reinterpret_cast<const uint32_t*>(&raw[u]));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int code = mx_block_code(amax);
        const float inv = mx_inv_scale(code);
        w[u].x = mx_encode4(v[0], v[1], v[2], v[3], inv);
        w[u].y = mx_encode4(v[4], v[5], v[6], v[7], inv);
        if (code == kMxNanScale) w[u] = make_uint2(kMxNanCodes, kMxNanCodes);
        if (part == 0 && b < nb) xs_tok[t * nb + b] = static_cast<uint8_t>(code);
      }
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_row, j);
        if (r < 0 || !dbg_row_ok(r, n_rows, err)) continue;   // warp-uniform
        uint8_t* dst = xq + static_cast<int64_t>(r) * H + part * 8;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int b = base + 8 * u + (lane >> 2);
          if (b < nb) *reinterpret_cast<uint2*>(dst + b * 32) = w[u];
        }
      }
    }
  }
}

cudaError_t launch_permute_quantize(const __nv_bfloat16* x, int64_t T, int H, int k,
                                    const int32_t* row_of, uint8_t* xq, uint8_t* xs_tok,
                                    cudaStream_t st, int64_t n_rows, int* err) {
  if (T == 0) return cudaSuccess;
  permute_quantize_kernel<<<grid_for_warps(T, 8), 256, 0, st>>>(x, T, H, k, row_of, xq, xs_tok,
                                                                 n_rows, err);
  return cudaGetLastError();
}

// One CTA per 128 permuted rows (one row block of the tiled layout). Each
// warp reads the token-order scale rows of 32 permuted rows (zeros for
// padding rows), 32 words of all 32 rows at a time with its lanes on
// consecutive words, so every load is one contiguous run of a row and 32 of
// them are in flight per lane. The words land row by row in shared memory
// with an odd row stride, and the CTA then writes the K/128 atoms (K/32 x
// 128 bytes) out contiguously, each thread assembling 16 bytes of an atom
// from four rows (atom word q holds row (q >> 2) + 32 (q & 3)).
// The odd stride keeps both the row writes and the atom reads free of bank
// conflicts.
__global__ void __launch_bounds__(128) gather_tile_scales_kernel(
    const uint8_t* __restrict__ xs_tok, const int32_t* __restrict__ token_of,
    const int32_t* __restrict__ off_al, const int32_t* __restrict__ counts, int E, int K,
    uint8_t* __restrict__ xs_tiled) {
  extern __shared__ uint32_t rows_w[];       // [128][stride] words
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTileM;
  if (r0 >= off_al[E]) return;               // capacity beyond the padded rows
  int lo = 0, hi = E - 1;                    // the expert that owns this row block
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off_al[mid] <= r0) lo = mid; else hi = mid - 1;
  }
  const int64_t real_end = static_cast<int64_t>(off_al[lo]) + counts[lo];
  const int kgroups = K >> 7, nb = K >> 5;
  const int stride = kgroups | 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t my_r = r0 + warp * 32 + lane;          // lane i: the token of row i
  const int my_tok = my_r < real_end ? __ldg(token_of + my_r) : -1;
  for (int c = 0; c < kgroups; c += 32) {              // 32 words of each of the 32 rows
    const int w = c + lane;
    uint32_t v[32];                                    // all 32 loads in flight at once
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int tok = __shfl_sync(0xffffffffu, my_tok, i);
      v[i] = (tok >= 0 && w < kgroups)
                 ? __ldg(reinterpret_cast<const uint32_t*>(xs_tok + static_cast<int64_t>(tok) * nb) + w)
                 : 0u;
    }
    if (w < kgroups) {
#pragma unroll
      for (int i = 0; i < 32; ++i) rows_w[(warp * 32 + i) * stride + w] = v[i];
    }
  }
  __syncthreads();
  int4* dst = reinterpret_cast<int4*>(xs_tiled + static_cast<int64_t>(blockIdx.x) * kgroups * 512);
  for (int j = threadIdx.x; j < kgroups * 32; j += blockDim.x) {
    const int kg = j >> 5, p = j & 31;       // atom kg, words 4p .. 4p + 3
    dst[j] = make_int4(static_cast<int>(rows_w[p * stride + kg]),
                       static_cast<int>(rows_w[(p + 32) * stride + kg]),
                       static_cast<int>(rows_w[(p + 64) * stride + kg]),
                       static_cast<int>(rows_w[(p + 96) * stride + kg]));
  }
}

cudaError_t launch_gather_tile_scales(const uint8_t* xs_tok, const int32_t* token_of,
                                      const int32_t* off_al, const int32_t* counts, int E, int K,
                                      int64_t cap, uint8_t* xs_tiled, cudaStream_t st) {
  const int smem = ((K >> 7) | 1) * kTileM * static_cast<int>(sizeof(uint32_t));
  static int configured[kMaxDevices] = {};    // per device: the largest size set so far
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return cudaErrorInvalidDevice;
  if (smem > 48 * 1024 && configured[d] < smem) {
    cudaError_t e = cudaFuncSetAttribute(gather_tile_scales_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[d] = smem;
  }
  gather_tile_scales_kernel<<<static_cast<unsigned>(cap / kTileM), kTileM, smem, st>>>(
      xs_tok, token_of, off_al, counts, E, K, xs_tiled);
  return cudaGetLastError();
}

// Row-major scales [rows, K/32] -> the tiled layout. One CTA per 128 output
// rows (one row block of atoms): thread i reads output row i's scale row
// (4 bytes at a time), drops the words into the block's atoms in shared
// memory, and the CTA writes the K/128 atoms out contiguously. With
// pair_half = P > 0, expert e has 2*rows_per_e virtual rows cut into tiles of
// 2P: row i of tile n is row n*P + i of src0 for i < P and row n*P + i - P of
// src1 otherwise (the gate | up halves of one fc1 N tile).
__global__ void __launch_bounds__(128) tile_scales_kernel(const uint8_t* __restrict__ src0,
                                                          const uint8_t* __restrict__ src1,
                                                          int64_t rows_per_e, int K,
                                                          int pair_half,
                                                          uint8_t* __restrict__ dst) {
  extern __shared__ uint32_t atoms[];        // [K/128][128] words
  const int i = threadIdx.x;
  const int64_t v = static_cast<int64_t>(blockIdx.x) * kTileM + i;
  const uint8_t* src = src0;
  int64_t srow = v;
  if (pair_half > 0) {
    const int64_t e = v / (2 * rows_per_e), vr = v - e * 2 * rows_per_e;
    const int64_t tile = vr / (2 * pair_half), in = vr - tile * 2 * pair_half;
    src = in < pair_half ? src0 : src1;
    srow = e * rows_per_e + tile * pair_half + (in < pair_half ? in : in - pair_half);
  }
  const int kgroups = K >> 7;
  const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src + srow * (K >> 5));
  const int word = (i & 31) * 4 + (i >> 5);
  for (int kg = 0; kg < kgroups; ++kg) atoms[kg * 128 + word] = __ldg(s32 + kg);
  __syncthreads();
  int4* out = reinterpret_cast<int4*>(dst + static_cast<int64_t>(blockIdx.x) * kgroups * 512);
  const int4* s4 = reinterpret_cast<const int4*>(atoms);
  for (int j = i; j < kgroups * 32; j += blockDim.x) out[j] = s4[j];
}

cudaError_t launch_tile_scales(const uint8_t* src0, const uint8_t* src1, int64_t out_rows,
                               int64_t rows_per_e, int K, int pair_half, uint8_t* dst,
                               cudaStream_t st) {
  if (out_rows == 0) return cudaSuccess;
  const int smem = (K >> 5) * kTileM;
  static int configured[kMaxDevices] = {};    // per device: the largest size set so far
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return cudaErrorInvalidDevice;
  if (smem > 48 * 1024 && configured[d] < smem) {
    cudaError_t e = cudaFuncSetAttribute(tile_scales_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[d] = smem;
  }
  tile_scales_kernel<<<static_cast<unsigned>(out_rows / kTileM), kTileM, smem, st>>>(
      src0, src1, rows_per_e, K, pair_half, dst);
  return cudaGetLastError();
}

}  // namespace moe
