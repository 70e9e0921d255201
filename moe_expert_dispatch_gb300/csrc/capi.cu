// capi.cu - the extern "C" entry points of include/moe_expert.h: argument
// checks, workspace layout, tensor-map encoding and the launch sequence of
// each call. No device memory is allocated here; every call is asynchronous.
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

// The device error word (one per device that loads the library). Kernels
// OR error bits into it; moe_get_error() reads and clears it.
__device__ int g_error_word;

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

namespace {

int* error_word() {
  static int* ptrs[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  if (!ptrs[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptrs[d] = static_cast<int*>(p);
  }
  return ptrs[d];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

// T * k < limit for k >= 1, without forming a product that could overflow.
bool rows_below(int64_t T, int k, int64_t limit) { return T <= (limit - 1) / k; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Forward workspace: byte offsets of every buffer.
struct FwdLayout {
  int64_t R, cap;
  size_t route, counts, offsets, off_al, row_of, token_of, prob_of, xp, h, o, ag, au, total;
};

FwdLayout fwd_layout(int64_t T, int H, int F, int E, int k, bool save) {
  FwdLayout L;
  L.R = T * k;
  L.cap = moe_padded_rows(L.R, E, kTileM);
  size_t cur = 0;
  auto take = [&](size_t bytes) {
    const size_t at = cur;
    cur += up256(bytes);
    return at;
  };
  L.route = take(route_scratch_bytes(L.R, E));
  L.counts = take(E * sizeof(int32_t));
  L.offsets = take((E + 1) * sizeof(int32_t));
  L.off_al = take((E + 1) * sizeof(int32_t));
  L.row_of = take(L.R * sizeof(int32_t));
  L.token_of = take(L.cap * sizeof(int32_t));
  L.prob_of = take(L.cap * sizeof(float));
  L.xp = take(static_cast<size_t>(L.cap) * H * 2);
  L.h = take(static_cast<size_t>(L.cap) * F * 2);
  L.o = take(static_cast<size_t>(L.cap) * H * 2);
  L.ag = save ? take(static_cast<size_t>(L.cap) * F * 2) : 0;
  L.au = save ? take(static_cast<size_t>(L.cap) * F * 2) : 0;
  L.total = cur;
  return L;
}

// Backward workspace: dO [cap, H] and dA = [dA_g | dA_u] [cap, 2F] in bf16 (GEMM
// operands), dXp [cap, H] in bf16 (a token's k rows summed in float into dX,
// then rounded once).
struct BwdLayout {
  int64_t cap;
  size_t d_o, d_a, d_xp, total;
};

BwdLayout bwd_layout(int64_t T, int H, int F, int E, int k) {
  BwdLayout B;
  B.cap = moe_padded_rows(T * k, E, kTileM);
  size_t cur = 0;
  auto take = [&](size_t bytes) {
    const size_t at = cur;
    cur += up256(bytes);
    return at;
  };
  B.d_o = take(static_cast<size_t>(B.cap) * H * 2);
  B.d_a = take(static_cast<size_t>(B.cap) * F * 2 * 2);
  B.d_xp = take(static_cast<size_t>(B.cap) * H * 2);
  B.total = cur;
  return B;
}

// MXFP8 forward workspace: the routing buffers of the BF16 layout, then the
// codes and tiled scales of x, the tiled scales of the weights, the codes
// and tiled scales of h, and O; with save_for_backward also A_g, A_u and h
// in bf16 [cap, F] (the backward's SwiGLU and weight-gradient operands).
struct MxLayout {
  int64_t R, cap;
  size_t route, counts, offsets, off_al, row_of, token_of, prob_of, xq, xs_tok, xs, wgu_s, wd_s,
      hq, hs, o, ag, au, hb, total;
};

MxLayout mx_layout(int64_t T, int H, int F, int E, int k, bool save = false) {
  MxLayout L;
  L.R = T * k;
  L.cap = moe_padded_rows(L.R, E, kTileM);
  size_t cur = 0;
  auto take = [&](size_t bytes) {
    const size_t at = cur;
    cur += up256(bytes);
    return at;
  };
  L.route = take(route_scratch_bytes(L.R, E));
  L.counts = take(E * sizeof(int32_t));
  L.offsets = take((E + 1) * sizeof(int32_t));
  L.off_al = take((E + 1) * sizeof(int32_t));
  L.row_of = take(L.R * sizeof(int32_t));
  L.token_of = take(L.cap * sizeof(int32_t));
  L.prob_of = take(L.cap * sizeof(float));
  L.xq = take(static_cast<size_t>(L.cap) * H);
  L.xs_tok = take(static_cast<size_t>(T) * H / 32);
  L.xs = take(static_cast<size_t>(L.cap) * H / 32);
  L.wgu_s = take(static_cast<size_t>(E) * 2 * F * H / 32);
  L.wd_s = take(static_cast<size_t>(E) * H * F / 32);
  L.hq = take(static_cast<size_t>(L.cap) * F);
  L.hs = take(static_cast<size_t>(L.cap) * F / 32);
  L.o = take(static_cast<size_t>(L.cap) * H * 2);
  L.ag = save ? take(static_cast<size_t>(L.cap) * F * 2) : 0;
  L.au = save ? take(static_cast<size_t>(L.cap) * F * 2) : 0;
  L.hb = save ? take(static_cast<size_t>(L.cap) * F * 2) : 0;
  L.total = cur;
  return L;
}

// MXFP8 backward workspace. Row-quantised operands of the data-gradient GEMMs
// (dO along H, dA along 2F) and column-quantised operands of the weight
// gradients ([C, cap], K = the padded rows), each with tiled scales; dXp in
// bf16; the weights' backward-orientation scales in the tiled layout.
struct MxBwdLayout {
  int64_t cap;
  size_t d_o, doq, dos, doT, dots, d_a, daq, das, daT, dats, d_xp, xpT, xpts, hT, hts, w2_st,
      w1g_st, w1u_st, total;
};

MxBwdLayout mx_bwd_layout(int64_t T, int H, int F, int E, int k) {
  MxBwdLayout L;
  L.cap = moe_padded_rows(T * k, E, kTileM);
  const size_t cap = static_cast<size_t>(L.cap);
  size_t cur = 0;
  auto take = [&](size_t bytes) {
    const size_t at = cur;
    cur += up256(bytes);
    return at;
  };
  L.d_o = take(cap * H * 2);
  L.doq = take(cap * H);
  L.dos = take(cap * H / 32);
  L.doT = take(cap * H);
  L.dots = take(cap * H / 32);
  L.d_a = take(cap * 2 * F * 2);
  L.daq = take(cap * 2 * F);
  L.das = take(cap * 2 * F / 32);
  L.daT = take(cap * 2 * F);
  L.dats = take(cap * 2 * F / 32);
  L.d_xp = take(cap * H * 2);
  L.xpT = take(cap * H);
  L.xpts = take(cap * H / 32);
  L.hT = take(cap * F);
  L.hts = take(cap * F / 32);
  L.w2_st = take(static_cast<size_t>(E) * F * H / 32);
  L.w1g_st = take(static_cast<size_t>(E) * H * F / 32);
  L.w1u_st = take(static_cast<size_t>(E) * H * F / 32);
  L.total = cur;
  return L;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

moe_config cfg_or_default(const moe_config* c) {
  moe_config d;
  moe_config_init(&d);
  if (!c) return d;
  d = *c;
  if (d.ring_stages < 0 || d.ring_stages > 6) d.ring_stages = 0;   // 0: the kernel's deepest
  if (d.wait_limit_ns <= 0) d.wait_limit_ns = static_cast<long long>(kDefaultWaitNs);
  return d;
}

// MMA N of the MXFP8 GEMMs: 256 halves the A traffic per FLOP; 128 keeps two
// accumulators (and is the only width when H is not a multiple of 256)
int mx_tile_n(const moe_config& c, int H, int F) {
  return c.mxfp8_tile_n == 128 ? 128
         : (c.mxfp8_tile_n == 256 || (F % 128 == 0 && H % 256 == 0)) ? 256 : 128;
}

moe_status check_block_args(int64_t T, int H, int F, int E, int k) {
  if (T < 0 || H <= 0 || F <= 0 || E < 1 || E > kMaxExperts || k < 1 || k > E || k > kMaxTopK)
    return MOE_ERR_INVALID_ARG;
  if (!rows_below(T, k, (static_cast<int64_t>(1) << 31) - kTileM * kMaxExperts))
    return MOE_ERR_INVALID_ARG;
  if (H % 128 != 0 || F % 128 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Operands at most this large are kept in L2 (evict_last) while a GEMM re-reads
// them across its N tiles; larger ones would only push the weights out.
constexpr uint64_t kKeepInL2Bytes = 96ull << 20;

int keep(uint64_t bytes) { return bytes <= kKeepInL2Bytes ? 1 : 0; }

// Six events of the micro-batch pipeline, per thread and device, created on
// the first pipelined call and kept for the life of the process; a call
// re-records them, which leaves the waits of an earlier call untouched.
cudaEvent_t* pipeline_events() {
  static thread_local cudaEvent_t pool[kMaxDevices][6];
  static thread_local bool made[kMaxDevices];
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
  if (!made[d]) {
    for (int i = 0; i < 6; ++i)
      if (cudaEventCreateWithFlags(&pool[d][i], cudaEventDisableTiming) != cudaSuccess)
        return nullptr;
    made[d] = true;
  }
  return pool[d];
}

// CTA pairs for the BF16 GEMMs over routed rows: as configured, else when
// the experts average at least 4 row blocks of 128, where the half-filled
// last tile of an expert with an odd block count costs little.
bool use_pairs(const moe_config& c, int64_t R, int E) {
  if (c.cta_pairs == 1) return false;
  if (c.cta_pairs == 2) return true;
  return R >= static_cast<int64_t>(4) * kTileM * E;
}

// Ring depth of the BF16 GEMMs: the configured one, capped at what fits
// (4 slots of 48 KB for one CTA per tile, 6 of 32 KB for a CTA of a pair).
int bf16_stages(const moe_config& c, bool pairs) {
  const int cap = pairs ? 6 : 4;
  return (c.ring_stages == 0 || c.ring_stages > cap) ? cap : c.ring_stages;
}

int grid_size(const moe_config& c) {
  const int sms = device_sm_count();
  return (c.num_sms > 0 && c.num_sms < sms) ? c.num_sms : sms;
}

}  // namespace

int* device_error_word() { return error_word(); }

int device_sm_count() {
  static int counts[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 1;
  if (!counts[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    counts[d] = n > 0 ? n : 1;
  }
  return counts[d];
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_scale_maps(MxScaleMaps* m, const uint8_t* sfa, uint64_t sfa_bytes, const uint8_t* sfb,
                     uint64_t sfb_bytes, const uint8_t* sfb1, uint64_t sfb1_bytes) {
  if (!make_tmap_scale_rows(&m->map[0], sfa, sfa_bytes) ||
      !make_tmap_scale_rows(&m->map[1], sfb, sfb_bytes))
    return false;
  if (!sfb1) {
    m->map[2] = m->map[1];
    return true;
  }
  return make_tmap_scale_rows(&m->map[2], sfb1, sfb1_bytes);
}

bool make_tmap_scale_rows(CUtensorMap* map, const void* base, uint64_t bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || bytes % 512 != 0 || bytes == 0) return false;
  const cuuint64_t dims[2] = {256, bytes / 256};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {256, 2};   // one 512-byte scale atom
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_out_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, bool f32) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {f32 ? 16u : 32u, 32u};   // one epilogue warp's 32 rows
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe

using namespace moe;

extern "C" {

void moe_config_init(moe_config* cfg) {
  if (!cfg) return;
  memset(cfg, 0, sizeof(*cfg));
  cfg->ring_stages = 0;
  cfg->wait_limit_ns = static_cast<long long>(kDefaultWaitNs);
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id outside [0, E)";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_TIMEOUT: return "in-kernel wait timed out";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_BOUNDS: return "row index outside its buffer (debug build)";
  }
  return "unknown status";
}

moe_status moe_get_error(void* stream) {
  MOE_ENTRY_RANGE();
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  const int zero = 0;
  if (v && cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v & kErrBadId) return MOE_ERR_BAD_EXPERT_ID;
  if (v & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (v & kErrBounds) return MOE_ERR_BOUNDS;
  return MOE_OK;
}

int moe_num_sms(void) { return device_sm_count(); }

int64_t moe_padded_rows(int64_t n_rows, int E, int row_align) {
  if (row_align <= 1) return n_rows;
  const int64_t worst = n_rows + static_cast<int64_t>(E) * (row_align - 1);
  return (worst + row_align - 1) / row_align * row_align;
}

size_t moe_counts_workspace_size(int64_t n_ids, int E) {
  if (n_ids < 0 || E < 1) return 0;
  return route_scratch_bytes(n_ids, E);
}

moe_status moe_counts(const int32_t* ids, int64_t n_ids, int E, int32_t* counts, int32_t* offsets,
                      void* workspace, size_t ws_bytes, void* stream) {
  MOE_ENTRY_RANGE();
  if (n_ids < 0 || E < 1 || E > kMaxExperts || n_ids >= (static_cast<int64_t>(1) << 31))
    return MOE_ERR_INVALID_ARG;
  if ((n_ids > 0 && !ids) || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < route_scratch_bytes(n_ids, E)) return MOE_ERR_WORKSPACE;
  RouteScratch s = route_scratch(workspace, n_ids, E);
  return from_cuda(launch_counts(ids, n_ids, E, 1, counts, offsets, nullptr, s, error_word(),
                                 static_cast<cudaStream_t>(stream)));
}

size_t moe_route_topk_workspace_size(int64_t T, int k, int E) {
  if (T < 0 || k < 1 || E < 1 || !rows_below(T, k, static_cast<int64_t>(1) << 31)) return 0;
  return route_scratch_bytes(T * k, E);
}

moe_status moe_route_topk(const float* logits, int64_t T, int E, int k, int32_t* expert_ids,
                          float* probs, int32_t* counts, int32_t* offsets, void* workspace,
                          size_t ws_bytes, void* stream) {
  MOE_ENTRY_RANGE();
  if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > E || k > kMaxTopK ||
      !rows_below(T, k, static_cast<int64_t>(1) << 31))
    return MOE_ERR_INVALID_ARG;
  if ((T > 0 && (!logits || !expert_ids || !probs)) || !counts || !offsets)
    return MOE_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < route_scratch_bytes(T * k, E) || !aligned16(workspace))
    return MOE_ERR_WORKSPACE;
  RouteScratch s = route_scratch(workspace, T * k, E);
  return from_cuda(launch_route_topk(logits, T, E, k, 1, expert_ids, probs, counts, offsets,
                                     nullptr, s, static_cast<cudaStream_t>(stream)));
}

size_t moe_permute_workspace_size(int64_t T, int k, int E) {
  if (T < 0 || k < 1 || E < 1 || !rows_below(T, k, static_cast<int64_t>(1) << 31)) return 0;
  return route_scratch_bytes(T * k, E);
}

moe_status moe_permute(const void* x, int64_t T, int64_t row_bytes, const int32_t* ids,
                       const float* probs, int k, int E, int row_align, void* x_perm,
                       int32_t* row_of, int32_t* token_of, float* prob_of, int32_t* offsets,
                       int32_t* counts, void* workspace, size_t ws_bytes, void* stream) {
  MOE_ENTRY_RANGE();
  if (T < 0 || k < 1 || k > kMaxTopK || k > E || E > kMaxExperts || row_bytes <= 0 ||
      row_bytes % 16 != 0 || row_align < 1 || !rows_below(T, k, static_cast<int64_t>(1) << 31))
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !ids || !x_perm || !row_of || !token_of || !offsets || !counts)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < route_scratch_bytes(T * k, E)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouteScratch s = route_scratch(workspace, T * k, E);
  int* err = error_word();
  // dense offsets are wanted when row_align == 1; otherwise the padded ones
  cudaError_t e;
  if (row_align == 1)
    e = launch_counts(ids, T * k, E, 1, counts, offsets, nullptr, s, err, st);
  else
    e = launch_counts(ids, T * k, E, row_align, counts, nullptr, offsets, s, err, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  // x_perm, token_of and prob_of hold the padded row count (moe_padded_rows)
  const int64_t cap = moe_padded_rows(T * k, E, row_align);
  e = launch_rowmap(ids, probs, T * k, k, E, s, row_of, token_of, prob_of, st, cap, err);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return from_cuda(launch_permute_copy(x, T, row_bytes, k, row_of, x_perm, st, cap, err));
}

moe_status moe_unpermute(const void* o_perm, const int32_t* row_of, const float* probs, int64_t T,
                         int k, int H, void* y, void* stream) {
  MOE_ENTRY_RANGE();
  if (T < 0 || k < 1 || k > kMaxTopK || H <= 0 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!o_perm || !row_of || !y || !aligned16(o_perm) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_unpermute(static_cast<const __nv_bfloat16*>(o_perm), row_of, probs, T, k,
                                    H, static_cast<__nv_bfloat16*>(y),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_quantize_mxfp8(const void* in, int64_t rows, int K, uint8_t* q, uint8_t* scales,
                              void* stream) {
  MOE_ENTRY_RANGE();
  if (rows < 0 || K <= 0 || K % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!in || !q || !scales || !aligned16(in) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_quantize_mxfp8(static_cast<const __nv_bfloat16*>(in), rows, K, q, scales,
                                         static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute_quantize_mxfp8(const void* x, int64_t T, int H, const int32_t* row_of,
                                      int k, uint8_t* xq, uint8_t* xs, void* stream) {
  MOE_ENTRY_RANGE();
  if (T < 0 || H <= 0 || H % 32 != 0 || k < 1 || k > kMaxTopK) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !row_of || !xq || !xs || !aligned16(x) || reinterpret_cast<uintptr_t>(xq) % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_permute_quantize(static_cast<const __nv_bfloat16*>(x), T, H, k, row_of,
                                           xq, xs, static_cast<cudaStream_t>(stream)));
}

size_t moe_workspace_size(int64_t T, int H, int F, int E, int k, const moe_config* cfg,
                          int for_backward) {
  if (check_block_args(T, H, F, E, k) != MOE_OK) return 0;
  const moe_config c = cfg_or_default(cfg);
  if (for_backward) return bwd_layout(T, H, F, E, k).total;
  return fwd_layout(T, H, F, E, k, c.save_for_backward != 0).total;
}

// One BF16 forward over T tokens in one workspace, in three phases that
// may run on different streams: route (gate or counts, row map, permute),
// gemms (fc1 + SwiGLU, fc2) and combine (unpermute). Routing comes either
// from expert_ids / probs, or, when logits is given, from the fused gate,
// which writes ids_out / probs_out.
struct FwdRun {
  const void *x, *w_gate, *w_up, *w_down;
  const int32_t* expert_ids;
  const float* probs;
  const float* logits;
  int32_t* ids_out;
  float* probs_out;
  int64_t T;
  int H, F, E, k;
  void* y;
  void* ws;
  moe_config c;
  bool save;
  FwdLayout L;

  void mark(int i, cudaStream_t st) const {
    if (c.step_events && i < c.num_step_events)
      cudaEventRecord(static_cast<cudaEvent_t>(c.step_events[i]), st);
  }
  const int32_t* ids() const { return logits ? ids_out : expert_ids; }
  const float* weights() const { return logits ? probs_out : probs; }

  moe_status route(cudaStream_t st) const {
    const RouteScratch rs = route_scratch(at<char>(ws, L.route), L.R, E);
    int32_t* counts = at<int32_t>(ws, L.counts);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* off_al = at<int32_t>(ws, L.off_al);
    int32_t* row_of = at<int32_t>(ws, L.row_of);
    int32_t* token_of = at<int32_t>(ws, L.token_of);
    float* prob_of = at<float>(ws, L.prob_of);
    __nv_bfloat16* xp = at<__nv_bfloat16>(ws, L.xp);
    // (gate ->) counts -> offsets -> row map -> permute (the dispatch)
    if (logits) {
      if (launch_route_topk(logits, T, E, k, kTileM, ids_out, probs_out, counts, offsets, off_al,
                            rs, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else if (launch_counts(expert_ids, L.R, E, kTileM, counts, offsets, off_al, rs,
                             error_word(), st) != cudaSuccess) {
      return MOE_ERR_CUDA;
    }
    if (launch_rowmap(ids(), weights(), L.R, k, E, rs, row_of, token_of, prob_of, st, L.cap,
                      error_word()) != cudaSuccess)
      return MOE_ERR_CUDA;
    // with the fused gather, fc1 reads the routed rows straight from x; the
    // permuted copy is still made when the backward needs it
    const bool gather = c.fuse_gather != 0;
    if ((!gather || save) &&
        launch_permute_copy(x, T, static_cast<int64_t>(H) * 2, k, row_of, xp, st, L.cap,
                            error_word()) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (save && launch_zero_padding(counts, off_al, E, static_cast<int64_t>(H) * 2, xp, token_of,
                                    prob_of, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }

  moe_status gemms(cudaStream_t st) const {
    const bool gather = c.fuse_gather != 0;
    __nv_bfloat16* xp = at<__nv_bfloat16>(ws, L.xp);
    __nv_bfloat16* h = at<__nv_bfloat16>(ws, L.h);
    __nv_bfloat16* o = at<__nv_bfloat16>(ws, L.o);
    CUtensorMap ta, tg, tu, th, td;
    const bool ta_ok =
        gather ? make_tmap_bf16_2d(&ta, x, H, T, static_cast<uint64_t>(H) * 2, 64, 1)
               : make_tmap_bf16_2d(&ta, xp, H, L.cap, static_cast<uint64_t>(H) * 2, 64, kTileM);
    if (!ta_ok ||
        !make_tmap_bf16_2d(&tg, w_gate, F, static_cast<uint64_t>(E) * H,
                           static_cast<uint64_t>(F) * 2, 64, 64) ||
        !make_tmap_bf16_2d(&tu, w_up, F, static_cast<uint64_t>(E) * H,
                           static_cast<uint64_t>(F) * 2, 64, 64) ||
        !make_tmap_bf16_2d(&th, h, F, L.cap, static_cast<uint64_t>(F) * 2, 64, kTileM) ||
        !make_tmap_bf16_2d(&td, w_down, H, static_cast<uint64_t>(E) * F,
                           static_cast<uint64_t>(H) * 2, 64, 64))
      return MOE_ERR_CUDA;
    GroupedGemmArgs g1{};
    g1.off_al = at<int32_t>(ws, L.off_al);
    g1.E = E;
    g1.K = H;
    g1.N = F;
    g1.bn = 256;                 // 128 gate + 128 up columns per N tile
    g1.pair = (!gather && use_pairs(c, L.R, E)) ? 1 : 0;
    g1.stages = bf16_stages(c, g1.pair != 0);
    g1.b_rows = H;
    g1.b_split = 1;
    g1.out = h;
    g1.ldo = F;
    g1.save_g = save ? at<__nv_bfloat16>(ws, L.ag) : nullptr;
    g1.save_u = save ? at<__nv_bfloat16>(ws, L.au) : nullptr;
    g1.err = error_word();
    g1.wait_ns = static_cast<unsigned long long>(c.wait_limit_ns);
    g1.gather_token = at<int32_t>(ws, L.token_of);
    g1.gather_x = static_cast<const __nv_bfloat16*>(x);
    g1.counts = at<int32_t>(ws, L.counts);
    g1.keep_a = keep(static_cast<uint64_t>(L.R) * H * 2);
    const int grid = grid_size(c);
    GemmOut o1, o2;
    if (!make_out_tmap(&o1.map[0], h, F, L.cap, static_cast<uint64_t>(F) * 2, false) ||
        !make_out_tmap(&o2.map[0], o, H, L.cap, static_cast<uint64_t>(H) * 2, false))
      return MOE_ERR_CUDA;
    o1.map[1] = o1.map[2] = o1.map[0];          // A_g, A_u leave as blocks (save_g, save_u)
    g1.ld_act = F;
    o2.map[1] = o2.map[2] = o2.map[0];
    if ((gather ? launch_fc1_swiglu_gather(ta, tg, tu, o1, g1, grid, st)
                : launch_fc1_swiglu(ta, tg, tu, o1, g1, grid, st)) != cudaSuccess)
      return MOE_ERR_CUDA;
    mark(2, st);
    GroupedGemmArgs g2 = g1;
    g2.K = F;
    g2.N = H;
    g2.bn = (H % 256 == 0) ? 256 : 128;
    g2.b_rows = F;
    g2.b_split = 0;
    g2.out = o;
    g2.ldo = H;
    g2.save_g = g2.save_u = nullptr;
    g2.keep_a = keep(static_cast<uint64_t>(L.R) * F * 2);
    g2.pair = use_pairs(c, L.R, E) ? 1 : 0;     // fc2 gathers nothing: pairs as usual
    g2.stages = bf16_stages(c, g2.pair != 0);
    if (launch_fc2(th, td, o2, g2, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }

  moe_status combine(cudaStream_t st) const {
    return from_cuda(launch_unpermute(at<__nv_bfloat16>(ws, L.o), at<int32_t>(ws, L.row_of),
                                      weights(), T, k, H, static_cast<__nv_bfloat16*>(y), st,
                                      L.cap, error_word()));
  }
};

// Argument checks shared by the forward entry points; fills r but its layout.
static moe_status fwd_prepare(FwdRun& r, const void* x, const void* w_gate, const void* w_up,
                              const void* w_down, const int32_t* expert_ids, const float* probs,
                              const float* logits, int32_t* ids_out, float* probs_out, int64_t T,
                              int H, int F, int E, int k, void* y, const moe_config* cfg) {
  moe_status s = check_block_args(T, H, F, E, k);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!x || !w_gate || !w_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (logits ? (!ids_out || !probs_out) : (!expert_ids || !probs)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  r.x = x;
  r.w_gate = w_gate;
  r.w_up = w_up;
  r.w_down = w_down;
  r.expert_ids = expert_ids;
  r.probs = probs;
  r.logits = logits;
  r.ids_out = ids_out;
  r.probs_out = probs_out;
  r.T = T;
  r.H = H;
  r.F = F;
  r.E = E;
  r.k = k;
  r.y = y;
  r.c = cfg_or_default(cfg);
  r.save = r.c.save_for_backward != 0;
  return MOE_OK;
}

static moe_status expert_forward_impl(const void* x, const void* w_gate, const void* w_up,
                                      const void* w_down, const int32_t* expert_ids,
                                      const float* probs, const float* logits, int32_t* ids_out,
                                      float* probs_out, int64_t T, int H, int F, int E, int k,
                                      void* y, void* workspace, size_t ws_bytes,
                                      const moe_config* cfg, void* stream) {
  FwdRun r{};
  moe_status s = fwd_prepare(r, x, w_gate, w_up, w_down, expert_ids, probs, logits, ids_out,
                             probs_out, T, H, F, E, k, y, cfg);
  if (s != MOE_OK || T == 0) return s;
  r.L = fwd_layout(T, H, F, E, k, r.save);
  if (!workspace || ws_bytes < r.L.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  r.ws = workspace;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  r.mark(0, st);
  if ((s = r.route(st)) != MOE_OK) return s;
  r.mark(1, st);
  if ((s = r.gemms(st)) != MOE_OK) return s;
  r.mark(3, st);
  s = r.combine(st);
  r.mark(4, st);
  return s;
}

moe_status moe_expert_forward(const void* x, const void* w_gate, const void* w_up,
                              const void* w_down, const int32_t* expert_ids, const float* probs,
                              int64_t T, int H, int F, int E, int k, void* y, void* workspace,
                              size_t ws_bytes, const moe_config* cfg, void* stream) {
  MOE_ENTRY_RANGE();
  return expert_forward_impl(x, w_gate, w_up, w_down, expert_ids, probs, nullptr, nullptr, nullptr,
                             T, H, F, E, k, y, workspace, ws_bytes, cfg, stream);
}

moe_status moe_expert_forward_from_logits(const void* x, const void* w_gate, const void* w_up,
                                          const void* w_down, const float* router_logits,
                                          int64_t T, int H, int F, int E, int k,
                                          int32_t* expert_ids, float* probs, void* y,
                                          void* workspace, size_t ws_bytes,
                                          const moe_config* cfg, void* stream) {
  MOE_ENTRY_RANGE();
  if (T > 0 && !router_logits) return MOE_ERR_INVALID_ARG;
  return expert_forward_impl(x, w_gate, w_up, w_down, nullptr, nullptr, router_logits, expert_ids,
                             probs, T, H, F, E, k, y, workspace, ws_bytes, cfg, stream);
}

size_t moe_workspace_size_pipelined(int64_t T, int H, int F, int E, int k, int n_chunks) {
  if (check_block_args(T, H, F, E, k) != MOE_OK || n_chunks < 1) return 0;
  const int64_t tc = T > 0 ? (T + n_chunks - 1) / n_chunks : 0;
  return 2 * up256(fwd_layout(tc, H, F, E, k, false).total);
}

moe_status moe_expert_forward_pipelined(const void* x, const void* w_gate, const void* w_up,
                                        const void* w_down, const int32_t* expert_ids,
                                        const float* probs, int64_t T, int H, int F, int E, int k,
                                        void* y, int n_chunks, void* workspace, size_t ws_bytes,
                                        const moe_config* cfg, void* stream, void* aux_stream) {
  MOE_ENTRY_RANGE();
  FwdRun base{};
  moe_status s = fwd_prepare(base, x, w_gate, w_up, w_down, expert_ids, probs, nullptr, nullptr,
                             nullptr, T, H, F, E, k, y, cfg);
  if (s != MOE_OK) return s;
  if (n_chunks < 1 || !aux_stream || aux_stream == stream) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (base.save) return MOE_ERR_UNSUPPORTED;   // the backward reads one whole-batch workspace
  const int64_t tc = (T + n_chunks - 1) / n_chunks;
  const int64_t chunks = (T + tc - 1) / tc;
  const size_t slot = up256(fwd_layout(tc, H, F, E, k, false).total);
  if (!workspace || ws_bytes < 2 * slot || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  cudaEvent_t* ev = pipeline_events();
  if (!ev) return MOE_ERR_CUDA;
  cudaEvent_t start = ev[0], ready[2] = {ev[1], ev[2]}, gemms_done[2] = {ev[3], ev[4]},
              aux_done = ev[5];
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t aux = static_cast<cudaStream_t>(aux_stream);
  base.c.step_events = nullptr;
  base.c.num_step_events = 0;
  auto chunk = [&](int64_t c) {
    FwdRun r = base;
    const int64_t t0 = c * tc;
    r.T = (T - t0 < tc) ? T - t0 : tc;
    r.x = static_cast<const char*>(x) + t0 * H * 2;
    r.expert_ids = expert_ids + t0 * k;
    r.probs = probs + t0 * k;
    r.y = static_cast<char*>(y) + t0 * H * 2;
    r.ws = static_cast<char*>(workspace) + (c & 1) * slot;
    r.L = fwd_layout(r.T, H, F, E, k, false);
    return r;
  };
  // aux: route(0) | route(c+1) while st runs the GEMMs of c | combine(c)
  // while st runs the GEMMs of c+1. Chunk c uses workspace slot c % 2; the
  // route of c+1 waits for the GEMMs of c-1 (the slot's last reader on st),
  // and the combine of c-1 precedes it on aux.
  if (cudaEventRecord(start, st) != cudaSuccess || cudaStreamWaitEvent(aux, start, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  if ((s = chunk(0).route(aux)) != MOE_OK) return s;
  if (cudaEventRecord(ready[0], aux) != cudaSuccess) return MOE_ERR_CUDA;
  for (int64_t c = 0; c < chunks; ++c) {
    const FwdRun r = chunk(c);
    if (cudaStreamWaitEvent(st, ready[c & 1], 0) != cudaSuccess) return MOE_ERR_CUDA;
    if ((s = r.gemms(st)) != MOE_OK) return s;
    if (cudaEventRecord(gemms_done[c & 1], st) != cudaSuccess) return MOE_ERR_CUDA;
    if (c + 1 < chunks) {
      const FwdRun next = chunk(c + 1);
      if (c >= 1 && cudaStreamWaitEvent(aux, gemms_done[(c + 1) & 1], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
      if ((s = next.route(aux)) != MOE_OK) return s;
      if (cudaEventRecord(ready[(c + 1) & 1], aux) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (cudaStreamWaitEvent(aux, gemms_done[c & 1], 0) != cudaSuccess) return MOE_ERR_CUDA;
    if ((s = r.combine(aux)) != MOE_OK) return s;
  }
  if (cudaEventRecord(aux_done, aux) != cudaSuccess ||
      cudaStreamWaitEvent(st, aux_done, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_expert_backward(const void* dy, const void* x, const void* w_gate, const void* w_up,
                               const void* w_down, const int32_t* expert_ids, const float* probs,
                               int64_t T, int H, int F, int E, int k, const void* fwd_ws,
                               size_t fwd_ws_bytes, void* dx, float* dw_gate, float* dw_up,
                               float* dw_down, float* dprobs, int accumulate_dw, void* workspace,
                               size_t ws_bytes, const moe_config* cfg, void* stream) {
  MOE_ENTRY_RANGE();
  moe_status s = check_block_args(T, H, F, E, k);
  if (s != MOE_OK) return s;
  if (!w_gate || !w_up || !w_down || !dw_gate || !dw_up || !dw_down) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(dw_gate) ||
      !aligned16(dw_up) || !aligned16(dw_down))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    // no tokens: every expert is empty, so the weight gradients are zero
    if (accumulate_dw) return MOE_OK;
    const size_t wb = static_cast<size_t>(E) * H * F * sizeof(float);
    if (cudaMemsetAsync(dw_gate, 0, wb, st) != cudaSuccess ||
        cudaMemsetAsync(dw_up, 0, wb, st) != cudaSuccess ||
        cudaMemsetAsync(dw_down, 0, wb, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  (void)x;
  (void)expert_ids;
  if (!dy || !probs || !dx || !dprobs || !fwd_ws || !aligned16(dy) || !aligned16(dx))
    return MOE_ERR_INVALID_ARG;
  const moe_config c = cfg_or_default(cfg);
  const FwdLayout L = fwd_layout(T, H, F, E, k, true);
  if (fwd_ws_bytes < L.total || !aligned16(fwd_ws)) return MOE_ERR_WORKSPACE;
  const BwdLayout B = bwd_layout(T, H, F, E, k);
  if (!workspace || ws_bytes < B.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  int* err = error_word();
  void* fw = const_cast<void*>(fwd_ws);
  const int32_t* counts = at<int32_t>(fw, L.counts);
  const int32_t* off_al = at<int32_t>(fw, L.off_al);
  const int32_t* row_of = at<int32_t>(fw, L.row_of);
  const __nv_bfloat16* xp = at<__nv_bfloat16>(fw, L.xp);
  const __nv_bfloat16* h = at<__nv_bfloat16>(fw, L.h);
  const __nv_bfloat16* o = at<__nv_bfloat16>(fw, L.o);
  const __nv_bfloat16* ag = at<__nv_bfloat16>(fw, L.ag);
  const __nv_bfloat16* au = at<__nv_bfloat16>(fw, L.au);
  __nv_bfloat16* d_o = at<__nv_bfloat16>(workspace, B.d_o);
  __nv_bfloat16* d_a = at<__nv_bfloat16>(workspace, B.d_a);
  __nv_bfloat16* d_xp = at<__nv_bfloat16>(workspace, B.d_xp);
  const int grid = grid_size(c);
  const int bnF = (F % 256 == 0) ? 256 : 128;
  const int bnH = (H % 256 == 0) ? 256 : 128;
  // dH and dXp run on CTA pairs as the forward does; a pair's CTA reads its
  // half of the K-major B tile, bn / 2 rows
  const bool pairs = use_pairs(c, T * k, E);
  const int bF = pairs ? bnF / 2 : bnF, bH = pairs ? bnH / 2 : bnH;
  auto mark = [&](int i) {
    if (c.step_events && i < c.num_step_events)
      cudaEventRecord(static_cast<cudaEvent_t>(c.step_events[i]), st);
  };
  mark(0);

  // dO = p dY (gather-scale) and dprobs = <dY, O>; padding rows of dO are zero
  if (launch_dout(static_cast<const __nv_bfloat16*>(dy), o, row_of, probs, T, k, H, d_o, dprobs,
                  st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_zero_padding(counts, off_al, E, static_cast<int64_t>(H) * 2, d_o, nullptr, nullptr,
                          st) != cudaSuccess)
    return MOE_ERR_CUDA;
  mark(1);

  CUtensorMap t_do, t_w2k, t_da, t_wgk, t_wuk, t_xp_mn, t_da_mn, t_h_mn, t_do_mn;
  if (!make_tmap_bf16_2d(&t_do, d_o, H, B.cap, static_cast<uint64_t>(H) * 2, 64, kTileM) ||
      !make_tmap_bf16_2d(&t_w2k, w_down, H, static_cast<uint64_t>(E) * F,
                         static_cast<uint64_t>(H) * 2, 64, bF) ||
      !make_tmap_bf16_2d(&t_da, d_a, 2 * static_cast<uint64_t>(F), B.cap,
                         static_cast<uint64_t>(F) * 4, 64, kTileM) ||
      !make_tmap_bf16_2d(&t_wgk, w_gate, F, static_cast<uint64_t>(E) * H,
                         static_cast<uint64_t>(F) * 2, 64, bH) ||
      !make_tmap_bf16_2d(&t_wuk, w_up, F, static_cast<uint64_t>(E) * H,
                         static_cast<uint64_t>(F) * 2, 64, bH) ||
      !make_tmap_bf16_2d(&t_xp_mn, xp, H, L.cap, static_cast<uint64_t>(H) * 2, 64, 64) ||
      !make_tmap_bf16_2d(&t_da_mn, d_a, 2 * static_cast<uint64_t>(F), B.cap,
                         static_cast<uint64_t>(F) * 4, 64, 64) ||
      !make_tmap_bf16_2d(&t_h_mn, h, F, L.cap, static_cast<uint64_t>(F) * 2, 64, 64) ||
      !make_tmap_bf16_2d(&t_do_mn, d_o, H, B.cap, static_cast<uint64_t>(H) * 2, 64, 64))
    return MOE_ERR_CUDA;

  // dH = dO W2^T, then dA_g, dA_u from the saved A_g, A_u
  GroupedGemmArgs g{};
  g.off_al = off_al;
  g.E = E;
  g.stages = bf16_stages(c, false);
  g.err = err;
  g.wait_ns = static_cast<unsigned long long>(c.wait_limit_ns);
  GroupedGemmArgs gh = g;
  gh.pair = pairs ? 1 : 0;
  gh.stages = bf16_stages(c, pairs);
  gh.K = H;
  gh.N = F;
  gh.bn = bnF;
  gh.b_rows = F;
  gh.out = d_a;
  gh.ldo = 2 * static_cast<int64_t>(F);
  gh.out_split = F;
  gh.act_g = ag;
  gh.act_u = au;
  gh.ld_act = F;
  gh.keep_a = keep(static_cast<uint64_t>(T) * k * H * 2);
  GemmOut oh, ox, ow1, ow2;
  if (!make_out_tmap(&oh.map[0], d_a, 2 * static_cast<uint64_t>(F), B.cap,
                     static_cast<uint64_t>(F) * 4, false) ||
      !make_out_tmap(&ox.map[0], d_xp, H, B.cap, static_cast<uint64_t>(H) * 2, false) ||
      !make_out_tmap(&ow1.map[0], dw_gate, F, static_cast<uint64_t>(E) * H,
                     static_cast<uint64_t>(F) * 4, true) ||
      !make_out_tmap(&ow1.map[1], dw_up, F, static_cast<uint64_t>(E) * H,
                     static_cast<uint64_t>(F) * 4, true) ||
      !make_out_tmap(&ow2.map[0], dw_down, H, static_cast<uint64_t>(E) * F,
                     static_cast<uint64_t>(H) * 4, true))
    return MOE_ERR_CUDA;
  oh.map[1] = oh.map[2] = oh.map[0];
  ox.map[1] = ox.map[2] = ox.map[0];
  ow1.map[2] = ow1.map[0];
  ow2.map[1] = ow2.map[2] = ow2.map[0];
  if (launch_dh_swiglu_bwd(t_do, t_w2k, oh, gh, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
  mark(2);

  // dXp = bf16(dA_g W1g^T + dA_u W1u^T) (one reduction over 2F), then
  // dX = bf16(sum_j dXp[row_of]), the combine with unit weights
  GroupedGemmArgs gx = g;
  gx.pair = pairs ? 1 : 0;
  gx.stages = bf16_stages(c, pairs);
  gx.K = 2 * F;
  gx.N = H;
  gx.bn = bnH;
  gx.b_rows = H;
  gx.b_split = 2;
  gx.k_split = F / 64;
  gx.out = d_xp;
  gx.ldo = H;
  gx.keep_a = keep(static_cast<uint64_t>(T) * k * F * 4);
  if (launch_dxp(t_da, t_wgk, t_wuk, ox, gx, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
  mark(3);
  if (launch_unpermute(d_xp, row_of, nullptr, T, k, H, static_cast<__nv_bfloat16*>(dx), st, L.cap,
                       err) != cudaSuccess)
    return MOE_ERR_CUDA;
  mark(4);

  // dW1g | dW1u = Xp_e^T [dA_g | dA_u] and dW2 = h_e^T dO_e over each expert's rows
  GroupedGemmArgs gw1 = g;
  gw1.pair = (pairs && H % 256 == 0) ? 1 : 0;      // the gradient's rows in M = 256 tiles
  gw1.stages = bf16_stages(c, gw1.pair != 0);
  gw1.M = H;
  gw1.N = 2 * F;
  gw1.bn = bnF;
  gw1.out_split = F;
  gw1.outf = dw_gate;
  gw1.outf2 = dw_up;
  gw1.accumulate = accumulate_dw ? 1 : 0;
  gw1.keep_a = keep(static_cast<uint64_t>(T) * k * H * 2);
  if (launch_wgrad(t_xp_mn, t_da_mn, ow1, gw1, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
  mark(5);
  GroupedGemmArgs gw2 = g;
  gw2.pair = (pairs && F % 256 == 0) ? 1 : 0;
  gw2.stages = bf16_stages(c, gw2.pair != 0);
  gw2.M = F;
  gw2.N = H;
  gw2.bn = bnH;
  gw2.out_split = 0;
  gw2.outf = dw_down;
  gw2.accumulate = accumulate_dw ? 1 : 0;
  gw2.keep_a = keep(static_cast<uint64_t>(T) * k * F * 2);
  if (launch_wgrad(t_h_mn, t_do_mn, ow2, gw2, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
  mark(6);
  return MOE_OK;
}

size_t moe_workspace_size_mxfp8(int64_t T, int H, int F, int E, int k, const moe_config* cfg) {
  if (check_block_args(T, H, F, E, k) != MOE_OK) return 0;
  const moe_config c = cfg_or_default(cfg);
  return mx_layout(T, H, F, E, k, c.save_for_backward != 0).total;
}

size_t moe_workspace_size_mxfp8_backward(int64_t T, int H, int F, int E, int k) {
  if (check_block_args(T, H, F, E, k) != MOE_OK) return 0;
  return mx_bwd_layout(T, H, F, E, k).total;
}

moe_status moe_quantize_mxfp8_dual(const void* in, int64_t batch, int rows, int cols,
                                   uint8_t* q_rows, uint8_t* s_rows, uint8_t* q_cols,
                                   uint8_t* s_cols, void* stream) {
  MOE_ENTRY_RANGE();
  if (batch < 0 || rows <= 0 || cols <= 0 || rows % 32 != 0 || cols % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (batch == 0) return MOE_OK;
  if (!in || !q_rows || !s_rows || !q_cols || !s_cols || !aligned16(in) || !aligned16(q_rows) ||
      !aligned16(q_cols))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_quantize_dual(static_cast<const __nv_bfloat16*>(in), cols, batch,
                                        static_cast<int64_t>(rows) * cols, rows, cols, nullptr,
                                        false, q_rows, s_rows, q_cols, s_cols,
                                        static_cast<cudaStream_t>(stream)));
}

moe_status moe_quantize_mxfp8_t(const void* in, int64_t batch, int rows, int cols, uint8_t* q,
                                uint8_t* scales, void* stream) {
  MOE_ENTRY_RANGE();
  if (batch < 0 || rows <= 0 || cols <= 0 || rows % 32 != 0 || cols % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  if (batch == 0) return MOE_OK;
  if (!in || !q || !scales || !aligned16(in) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_quantize_cols(static_cast<const __nv_bfloat16*>(in), cols, batch,
                                        static_cast<int64_t>(rows) * cols, rows, cols, nullptr, 0,
                                        nullptr, false, q, scales,
                                        static_cast<cudaStream_t>(stream)));
}

moe_status moe_tile_weight_scales_mxfp8(const uint8_t* wg_s, const uint8_t* wu_s,
                                        const uint8_t* wd_s, int H, int F, int E,
                                        const moe_config* cfg, uint8_t* wgu_tiled,
                                        uint8_t* wd_tiled, void* stream) {
  MOE_ENTRY_RANGE();
  moe_status s = check_block_args(0, H, F, E, 1);
  if (s != MOE_OK) return s;
  if (!wg_s || !wu_s || !wd_s || !wgu_tiled || !wd_tiled) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(wg_s) & 3) || (reinterpret_cast<uintptr_t>(wu_s) & 3) ||
      (reinterpret_cast<uintptr_t>(wd_s) & 3) || !aligned16(wgu_tiled) || !aligned16(wd_tiled))
    return MOE_ERR_INVALID_ARG;
  const moe_config c = cfg_or_default(cfg);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_tile_scales(wg_s, wu_s, static_cast<int64_t>(E) * 2 * F, F, H, mx_tile_n(c, H, F) / 2,
                         wgu_tiled, st) != cudaSuccess ||
      launch_tile_scales(wd_s, nullptr, static_cast<int64_t>(E) * H, H, F, 0, wd_tiled, st) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_expert_forward_mxfp8(const void* x, const uint8_t* wg_q, const uint8_t* wg_s,
                                    const uint8_t* wu_q, const uint8_t* wu_s, const uint8_t* wd_q,
                                    const uint8_t* wd_s, const int32_t* expert_ids,
                                    const float* probs, int64_t T, int H, int F, int E, int k,
                                    void* y, void* workspace, size_t ws_bytes,
                                    const moe_config* cfg, void* stream) {
  MOE_ENTRY_RANGE();
  moe_status s = check_block_args(T, H, F, E, k);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  const moe_config c = cfg_or_default(cfg);
  const bool pretiled = c.mx_scales_pretiled != 0;
  if (!x || !wg_q || !wg_s || !wu_q || (!wu_s && !pretiled) || !wd_q || !wd_s || !expert_ids ||
      !probs || !y)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(wg_q) || !aligned16(wu_q) || !aligned16(wd_q) ||
      !aligned16(y) || (reinterpret_cast<uintptr_t>(wg_s) & 3) ||
      (!pretiled && (reinterpret_cast<uintptr_t>(wu_s) & 3)) ||
      (reinterpret_cast<uintptr_t>(wd_s) & 3) ||
      (pretiled && (!aligned16(wg_s) || !aligned16(wd_s))))   // read by bulk copies
    return MOE_ERR_INVALID_ARG;
  const bool save = c.save_for_backward != 0;
  const MxLayout L = mx_layout(T, H, F, E, k, save);
  if (!workspace || ws_bytes < L.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = error_word();
  auto mark = [&](int i) {
    if (c.step_events && i < c.num_step_events)
      cudaEventRecord(static_cast<cudaEvent_t>(c.step_events[i]), st);
  };
  mark(0);
  const RouteScratch rs = route_scratch(at<char>(workspace, L.route), L.R, E);
  int32_t* counts = at<int32_t>(workspace, L.counts);
  int32_t* offsets = at<int32_t>(workspace, L.offsets);
  int32_t* off_al = at<int32_t>(workspace, L.off_al);
  int32_t* row_of = at<int32_t>(workspace, L.row_of);
  int32_t* token_of = at<int32_t>(workspace, L.token_of);
  float* prob_of = at<float>(workspace, L.prob_of);
  uint8_t* xq = at<uint8_t>(workspace, L.xq);
  uint8_t* xs_tok = at<uint8_t>(workspace, L.xs_tok);
  uint8_t* xs = at<uint8_t>(workspace, L.xs);
  // the weights' scales in the block-scaled MMA's layout: given, or tiled here
  const uint8_t* wgu_s = pretiled ? wg_s : at<uint8_t>(workspace, L.wgu_s);
  const uint8_t* wd_st = pretiled ? wd_s : at<uint8_t>(workspace, L.wd_s);
  uint8_t* hq = at<uint8_t>(workspace, L.hq);
  uint8_t* hs = at<uint8_t>(workspace, L.hs);
  __nv_bfloat16* o = at<__nv_bfloat16>(workspace, L.o);

  // counts -> offsets -> row map -> permute + quantise x (the dispatch)
  if (launch_counts(expert_ids, L.R, E, kTileM, counts, offsets, off_al, rs, err, st) !=
          cudaSuccess ||
      launch_rowmap(expert_ids, probs, L.R, k, E, rs, row_of, token_of, prob_of, st, L.cap,
                    err) != cudaSuccess ||
      launch_permute_quantize(static_cast<const __nv_bfloat16*>(x), T, H, k, row_of, xq, xs_tok,
                              st, L.cap, err) != cudaSuccess ||
      launch_gather_tile_scales(xs_tok, token_of, off_al, counts, E, H, L.cap, xs, st) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  // the backward reads the padding rows as zeros (their h is then zero) and
  // marks them in token_of
  if (save && launch_zero_padding(counts, off_al, E, H, xq, token_of, prob_of, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int mx_bn = mx_tile_n(c, H, F);
  if (!pretiled &&
      (launch_tile_scales(wg_s, wu_s, static_cast<int64_t>(E) * 2 * F, F, H, mx_bn / 2,
                          at<uint8_t>(workspace, L.wgu_s), st) != cudaSuccess ||
       launch_tile_scales(wd_s, nullptr, static_cast<int64_t>(E) * H, H, F, 0,
                          at<uint8_t>(workspace, L.wd_s), st) != cudaSuccess))
    return MOE_ERR_CUDA;
  mark(1);

  // CTA pairs only when asked for: measured on the MXFP8 workloads they are
  // no faster (the pair's copies of the scale atoms into tensor memory cost
  // it about a fifth of its tensor pipe). A pair's CTA reads N / 2 rows of B.
  const bool pairs = c.cta_pairs == 2;
  const uint32_t b_box = (pairs && mx_bn == 128) ? 64 : 128;
  CUtensorMap ta, tg, tu, th, td;
  if (!make_tmap_u8_2d(&ta, xq, H, L.cap, H, 128, kTileM) ||
      !make_tmap_u8_2d(&tg, wg_q, H, static_cast<uint64_t>(E) * F, H, 128, mx_bn / 2) ||
      !make_tmap_u8_2d(&tu, wu_q, H, static_cast<uint64_t>(E) * F, H, 128, mx_bn / 2) ||
      !make_tmap_u8_2d(&th, hq, F, L.cap, F, 128, kTileM) ||
      !make_tmap_u8_2d(&td, wd_q, F, static_cast<uint64_t>(E) * H, F, 128, b_box))
    return MOE_ERR_CUDA;
  const int grid = grid_size(c);
  MxGemmArgs g1{};
  g1.off_al = off_al;
  g1.E = E;
  g1.K = H;
  g1.N = F;
  g1.stages = c.ring_stages == 0 ? 6 : c.ring_stages;
  g1.bn = mx_bn;
  g1.keep_a = keep(static_cast<uint64_t>(L.R) * H);
  g1.b_rows = F;
  g1.sfb_rows = 2 * static_cast<int64_t>(F);
  g1.sfa = xs;
  g1.sfb = wgu_s;
  g1.hq = hq;
  g1.hs = hs;
  GemmOut o1, o2;
  g1.save = save ? 1 : 0;
  if (save) {   // A_g, A_u and h in bf16, blocked, for the backward
    g1.save_g = at<__nv_bfloat16>(workspace, L.ag);
    g1.save_u = at<__nv_bfloat16>(workspace, L.au);
    g1.save_h = at<__nv_bfloat16>(workspace, L.hb);
    o1.map[0] = o1.map[1] = o1.map[2] = ta;    // unused
  } else {
    o1.map[0] = o1.map[1] = o1.map[2] = ta;    // unused
  }
  g1.err = err;
  g1.wait_ns = static_cast<unsigned long long>(c.wait_limit_ns);
  g1.pair = pairs ? 1 : 0;
  MxScaleMaps s1, s2;
  if (!make_scale_maps(&s1, xs, static_cast<uint64_t>(L.cap) * H / 32, wgu_s,
                       static_cast<uint64_t>(E) * 2 * F * H / 32) ||
      !make_scale_maps(&s2, hs, static_cast<uint64_t>(L.cap) * F / 32, wd_st,
                       static_cast<uint64_t>(E) * H * F / 32))
    return MOE_ERR_CUDA;
  if (launch_mx_fc1(ta, tg, tu, o1, g1, grid, st, s1) != cudaSuccess)
    return MOE_ERR_CUDA;
  mark(2);
  MxGemmArgs g2 = g1;
  g2.K = F;
  g2.N = H;
  g2.b_rows = H;
  g2.sfb_rows = H;
  g2.sfa = hs;
  g2.sfb = wd_st;
  g2.keep_a = keep(static_cast<uint64_t>(L.R) * F);
  g2.hq = nullptr;
  g2.hs = nullptr;
  g2.save = 0;
  if (!make_out_tmap(&o2.map[0], o, H, L.cap, static_cast<uint64_t>(H) * 2, false))
    return MOE_ERR_CUDA;
  o2.map[1] = o2.map[2] = o2.map[0];
  if (launch_mx_fc2(th, td, o2, g2, grid, st, s2) != cudaSuccess)
    return MOE_ERR_CUDA;
  mark(3);
  const cudaError_t ue =
      launch_unpermute(o, row_of, probs, T, k, H, static_cast<__nv_bfloat16*>(y), st, L.cap, err);
  mark(4);
  return from_cuda(ue);
}

moe_status moe_expert_backward_mxfp8(const void* dy, const void* x, const uint8_t* w1g_q,
                                     const uint8_t* w1g_s, const uint8_t* w1u_q,
                                     const uint8_t* w1u_s, const uint8_t* w2_q,
                                     const uint8_t* w2_s, const int32_t* expert_ids,
                                     const float* probs, int64_t T, int H, int F, int E, int k,
                                     const void* fwd_ws, size_t fwd_ws_bytes, void* dx,
                                     float* dw_gate_t, float* dw_up_t, float* dw_down_t,
                                     float* dprobs, int accumulate_dw, void* workspace,
                                     size_t ws_bytes, const moe_config* cfg, void* stream) {
  MOE_ENTRY_RANGE();
  moe_status s = check_block_args(T, H, F, E, k);
  if (s != MOE_OK) return s;
  if (!dw_gate_t || !dw_up_t || !dw_down_t || !aligned16(dw_gate_t) || !aligned16(dw_up_t) ||
      !aligned16(dw_down_t))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    // no tokens: every expert is empty, so the weight gradients are zero
    if (accumulate_dw) return MOE_OK;
    const size_t wb = static_cast<size_t>(E) * H * F * sizeof(float);
    if (cudaMemsetAsync(dw_gate_t, 0, wb, st) != cudaSuccess ||
        cudaMemsetAsync(dw_up_t, 0, wb, st) != cudaSuccess ||
        cudaMemsetAsync(dw_down_t, 0, wb, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  (void)expert_ids;
  if (!dy || !x || !probs || !dx || !dprobs || !fwd_ws || !w1g_q || !w1g_s || !w1u_q || !w1u_s ||
      !w2_q || !w2_s)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(dx) || !aligned16(w1g_q) ||
      !aligned16(w1u_q) || !aligned16(w2_q))
    return MOE_ERR_INVALID_ARG;
  const moe_config c = cfg_or_default(cfg);
  const MxLayout L = mx_layout(T, H, F, E, k, true);
  if (fwd_ws_bytes < L.total || !aligned16(fwd_ws)) return MOE_ERR_WORKSPACE;
  const MxBwdLayout B = mx_bwd_layout(T, H, F, E, k);
  if (!workspace || ws_bytes < B.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  void* fw = const_cast<void*>(fwd_ws);
  void* ws = workspace;
  const int32_t* counts = at<int32_t>(fw, L.counts);
  const int32_t* off_al = at<int32_t>(fw, L.off_al);
  const int32_t* row_of = at<int32_t>(fw, L.row_of);
  const int32_t* token_of = at<int32_t>(fw, L.token_of);
  const int32_t* row_end = off_al + E;          // rows past it are unused capacity
  const __nv_bfloat16* o = at<__nv_bfloat16>(fw, L.o);
  const __nv_bfloat16* ag = at<__nv_bfloat16>(fw, L.ag);
  const __nv_bfloat16* au = at<__nv_bfloat16>(fw, L.au);
  const __nv_bfloat16* hb = at<__nv_bfloat16>(fw, L.hb);
  const int64_t cap = B.cap;
  __nv_bfloat16* d_o = at<__nv_bfloat16>(ws, B.d_o);
  __nv_bfloat16* d_a = at<__nv_bfloat16>(ws, B.d_a);
  __nv_bfloat16* d_xp = at<__nv_bfloat16>(ws, B.d_xp);
  const int grid = grid_size(c);
  auto bn_for = [&](int n) {      // MMA N: the configured width when it divides n
    const int want = (c.mxfp8_tile_n == 128 || c.mxfp8_tile_n == 256) ? c.mxfp8_tile_n : 256;
    return n % want == 0 ? want : 128;
  };
  auto mark = [&](int i) {
    if (c.step_events && i < c.num_step_events)
      cudaEventRecord(static_cast<cudaEvent_t>(c.step_events[i]), st);
  };
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  mark(0);

  // dO = bf16(p dY) per routed row and dprobs = <dY, O>; padding rows of dO
  // are zero. dO quantised along H (dH's K) and along the rows (dW2's K).
  if (!ok(launch_dout(static_cast<const __nv_bfloat16*>(dy), o, row_of, probs, T, k, H, d_o,
                      dprobs, st)) ||
      !ok(launch_zero_padding(counts, off_al, E, static_cast<int64_t>(H) * 2, d_o, nullptr,
                              nullptr, st)) ||
      !ok(launch_quantize_dual(d_o, H, 1, 0, static_cast<int>(cap), H, row_end, true,
                               at<uint8_t>(ws, B.doq), at<uint8_t>(ws, B.dos),
                               at<uint8_t>(ws, B.doT), at<uint8_t>(ws, B.dots), st)) ||
      // the weights' backward-orientation scales in the MMA's tiled layout
      !ok(launch_tile_scales(w2_s, nullptr, static_cast<int64_t>(E) * F, F, H, 0,
                             at<uint8_t>(ws, B.w2_st), st)) ||
      !ok(launch_tile_scales(w1g_s, nullptr, static_cast<int64_t>(E) * H, H, F, 0,
                             at<uint8_t>(ws, B.w1g_st), st)) ||
      !ok(launch_tile_scales(w1u_s, nullptr, static_cast<int64_t>(E) * H, H, F, 0,
                             at<uint8_t>(ws, B.w1u_st), st)))
    return MOE_ERR_CUDA;
  mark(1);

  const int bnF = bn_for(F), bnH = bn_for(H);
  // dH and dXp on CTA pairs when asked for (a pair's CTA reads N / 2 rows of
  // B; the scale atoms arrive by tensor map)
  const bool pairs = c.cta_pairs == 2;
  const uint32_t box_f = (pairs && bnF == 128) ? 64 : 128;
  const uint32_t box_h = (pairs && bnH == 128) ? 64 : 128;
  CUtensorMap t_doq, t_w2, t_daq, t_w1g, t_w1u, t_daT, t_xpT, t_doT, t_hT;
  if (!make_tmap_u8_2d(&t_doq, at<uint8_t>(ws, B.doq), H, cap, H, 128, kTileM) ||
      !make_tmap_u8_2d(&t_w2, w2_q, H, static_cast<uint64_t>(E) * F, H, 128, box_f) ||
      !make_tmap_u8_2d(&t_daq, at<uint8_t>(ws, B.daq), 2 * static_cast<uint64_t>(F), cap,
                       2 * static_cast<uint64_t>(F), 128, kTileM) ||
      !make_tmap_u8_2d(&t_w1g, w1g_q, F, static_cast<uint64_t>(E) * H, F, 128, box_h) ||
      !make_tmap_u8_2d(&t_w1u, w1u_q, F, static_cast<uint64_t>(E) * H, F, 128, box_h) ||
      !make_tmap_u8_2d(&t_daT, at<uint8_t>(ws, B.daT), cap, 2 * static_cast<uint64_t>(F), cap,
                       128, kTileM) ||
      !make_tmap_u8_2d(&t_xpT, at<uint8_t>(ws, B.xpT), cap, H, cap, 128, 128) ||
      !make_tmap_u8_2d(&t_doT, at<uint8_t>(ws, B.doT), cap, H, cap, 128, kTileM) ||
      !make_tmap_u8_2d(&t_hT, at<uint8_t>(ws, B.hT), cap, F, cap, 128, 128))
    return MOE_ERR_CUDA;
  MxGemmArgs base{};
  base.off_al = off_al;
  base.E = E;
  base.stages = c.ring_stages == 0 ? 6 : c.ring_stages;
  base.err = error_word();
  base.wait_ns = static_cast<unsigned long long>(c.wait_limit_ns);

  // dH = deq(dO) deq(W2)^T over K = H, then the SwiGLU backward on the
  // saved A_g, A_u -> dA = [dA_g | dA_u] in bf16
  MxGemmArgs g = base;
  g.K = H;
  g.N = F;
  g.bn = bnF;
  g.b_rows = F;
  g.sfb_rows = F;
  g.sfa = at<uint8_t>(ws, B.dos);
  g.sfb = at<uint8_t>(ws, B.w2_st);
  g.act_g = ag;
  g.act_u = au;
  g.out_b = d_a;                                 // [dA_g | dA_u], blocked
  GemmOut od;
  od.map[0] = od.map[1] = od.map[2] = t_doq;     // unused
  g.keep_a = keep(static_cast<uint64_t>(cap) * H);
  MxScaleMaps sh, sx, sw1, sw2;
  if (!make_scale_maps(&sh, at<uint8_t>(ws, B.dos), static_cast<uint64_t>(cap) * H / 32,
                       at<uint8_t>(ws, B.w2_st), static_cast<uint64_t>(E) * F * H / 32) ||
      !make_scale_maps(&sx, at<uint8_t>(ws, B.das), static_cast<uint64_t>(cap) * 2 * F / 32,
                       at<uint8_t>(ws, B.w1g_st), static_cast<uint64_t>(E) * H * F / 32,
                       at<uint8_t>(ws, B.w1u_st), static_cast<uint64_t>(E) * H * F / 32) ||
      !make_scale_maps(&sw1, at<uint8_t>(ws, B.dats), static_cast<uint64_t>(cap) * 2 * F / 32,
                       at<uint8_t>(ws, B.xpts), static_cast<uint64_t>(cap) * H / 32) ||
      !make_scale_maps(&sw2, at<uint8_t>(ws, B.dots), static_cast<uint64_t>(cap) * H / 32,
                       at<uint8_t>(ws, B.hts), static_cast<uint64_t>(cap) * F / 32))
    return MOE_ERR_CUDA;
  const bool pair_h = pairs, pair_x = pairs;
  g.pair = pair_h ? 1 : 0;
  if (!ok(launch_mx_dh(t_doq, t_w2, od, g, grid, st, sh)))
    return MOE_ERR_CUDA;
  mark(2);

  // dA quantised along 2F (dXp's K) and along the rows (dW1's K)
  if (!ok(launch_quantize_dual_blocked(d_a, static_cast<int>(cap), 2 * F, row_end,
                                       at<uint8_t>(ws, B.daq), at<uint8_t>(ws, B.das),
                                       at<uint8_t>(ws, B.daT), at<uint8_t>(ws, B.dats), st)))
    return MOE_ERR_CUDA;
  mark(3);

  // dXp = bf16(deq(dA_g) deq(W1g)^T + deq(dA_u) deq(W1u)^T): K = 2F, the
  // first F from W1g, the second from W1u
  g = base;
  g.K = 2 * F;
  g.N = H;
  g.bn = bnH;
  g.b_rows = H;
  g.sfb_rows = H;
  g.k_split = F / 128;
  g.kgroups_b = F / 128;
  g.sfa = at<uint8_t>(ws, B.das);
  g.sfb = at<uint8_t>(ws, B.w1g_st);
  g.sfb1 = at<uint8_t>(ws, B.w1u_st);
  GemmOut ox;
  if (!make_out_tmap(&ox.map[0], d_xp, H, cap, static_cast<uint64_t>(H) * 2, false))
    return MOE_ERR_CUDA;
  ox.map[1] = ox.map[2] = ox.map[0];
  g.keep_a = keep(static_cast<uint64_t>(cap) * 2 * F);
  g.pair = pair_x ? 1 : 0;
  if (!ok(launch_mx_dxp(t_daq, t_w1g, t_w1u, ox, g, grid, st, sx)))
    return MOE_ERR_CUDA;
  mark(4);
  if (!ok(launch_unpermute(d_xp, row_of, nullptr, T, k, H, static_cast<__nv_bfloat16*>(dx), st,
                           cap, error_word())))
    return MOE_ERR_CUDA;
  mark(5);

  // weight gradients: x's routed rows and h quantised along the rows, then
  // dW1^T = deq(dA)^T deq(Xp) (rows 0..F-1 -> dw_gate_t, F..2F-1 -> dw_up_t)
  // and dW2^T = deq(dO)^T deq(h), K = each expert's padded rows
  if (!ok(launch_quantize_cols(static_cast<const __nv_bfloat16*>(x), H, 1, 0,
                               static_cast<int>(cap), H, token_of, T, row_end, true,
                               at<uint8_t>(ws, B.xpT), at<uint8_t>(ws, B.xpts), st)) ||
      !ok(launch_quantize_cols_blocked(hb, static_cast<int>(cap), F, row_end,
                                       at<uint8_t>(ws, B.hT), at<uint8_t>(ws, B.hts), st)))
    return MOE_ERR_CUDA;
  mark(6);
  const int kg_cap = static_cast<int>(cap / 128);
  g = base;
  g.M = 2 * F;
  g.N = H;
  g.bn = bnH;
  g.kgroups_a = kg_cap;
  g.kgroups_b = kg_cap;
  g.sfa = at<uint8_t>(ws, B.dats);
  g.sfb = at<uint8_t>(ws, B.xpts);
  GemmOut ow1, ow2;
  if (!make_out_tmap(&ow1.map[0], dw_gate_t, H, static_cast<uint64_t>(E) * F,
                     static_cast<uint64_t>(H) * 4, true) ||
      !make_out_tmap(&ow1.map[1], dw_up_t, H, static_cast<uint64_t>(E) * F,
                     static_cast<uint64_t>(H) * 4, true) ||
      !make_out_tmap(&ow2.map[0], dw_down_t, F, static_cast<uint64_t>(E) * H,
                     static_cast<uint64_t>(F) * 4, true))
    return MOE_ERR_CUDA;
  ow1.map[2] = ow1.map[0];
  ow2.map[1] = ow2.map[2] = ow2.map[0];
  g.out_split = F;
  g.accumulate = accumulate_dw;
  if (!ok(launch_mx_wgrad(t_daT, t_xpT, ow1, g, grid, st, sw1))) return MOE_ERR_CUDA;
  mark(7);
  g = base;
  g.M = H;
  g.N = F;
  g.bn = bnF;
  g.kgroups_a = kg_cap;
  g.kgroups_b = kg_cap;
  g.sfa = at<uint8_t>(ws, B.dots);
  g.sfb = at<uint8_t>(ws, B.hts);

  g.out_split = 0;
  g.accumulate = accumulate_dw;
  if (!ok(launch_mx_wgrad(t_doT, t_hT, ow2, g, grid, st, sw2))) return MOE_ERR_CUDA;
  mark(8);
  return MOE_OK;
}

}  // extern "C"
