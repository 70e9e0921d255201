// mx.cuh - MXFP8 (OCP Microscaling v1.0, E4M3 elements, E8M0 scales) on the
// device: the block quantiser's steps (scale exponent, inverse scale, E4M3
// encoding) shared by the standalone quantisers, the fused permute+quantise
// kernel and the fc1 epilogue, and the tiled scale layout that the
// block-scaled tensor-core MMA reads.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// floor(log2(a)) of a positive finite float, subnormals included.
__device__ __forceinline__ int floor_log2_pos(float a) {
  const uint32_t b = __float_as_uint(a);
  const int ex = static_cast<int>((b >> 23) & 0xFF);
  if (ex != 0) return ex - 127;
  const uint32_t man = b & 0x7FFFFF;
  return (31 - __clz(static_cast<int>(man))) - 149;
}

// Exponent s of the shared scale X = 2^s of a block whose largest magnitude
// is amax: floor(log2 amax) - 8, clamped to [-127, 127]; an all-zero block
// gets -127. The E8M0 code is s + 127.
__device__ __forceinline__ int mx_block_exp(float amax) {
  const int s = (amax > 0.0f) ? floor_log2_pos(amax) - 8 : -127;
  return max(-127, min(127, s));
}

// The bits of |v| as a float. Non-negative floats order like their bit
// patterns read as integers, and every infinity or NaN pattern (0x7F800000
// and above) lies above every finite one, so the integer maximum of these
// over a block is the bits of its largest magnitude, or a non-finite
// pattern when the block holds an infinity or a NaN (which fmaxf would drop).
__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// abs_bits of the largest magnitude among the 2n bf16 values packed in
// w[0..n): the sign bits cleared, each word's two halves compared as
// unsigned 16-bit numbers (which order like the magnitudes, with every
// infinity or NaN above every finite value), two values per instruction.
template <int n>
__device__ __forceinline__ uint32_t bf16x2_absmax_bits(const uint32_t* w) {
  uint32_t m = w[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int j = 1; j < n; ++j) m = __vmaxu2(m, w[j] & 0x7FFF7FFFu);
  return max(m & 0xFFFFu, m >> 16) << 16;   // bf16 bits to float bits
}

// A block that holds an infinity or a NaN has no finite shared scale: it is
// given the E8M0 NaN code and E4M3 NaN elements, so that every element of it
// decodes to NaN.
constexpr int kMxNanScale = 0xFF;
constexpr uint32_t kMxNanCodes = 0x7F7F7F7Fu;   // four E4M3 NaNs (S.1111.111, S = 0)

// E8M0 code of the block whose largest magnitude has the bits amax_bits
// (see abs_bits): mx_block_exp + 127, or kMxNanScale for a non-finite block.
__device__ __forceinline__ int mx_block_code(uint32_t amax_bits) {
  return amax_bits >= 0x7F800000u ? kMxNanScale : mx_block_exp(__uint_as_float(amax_bits)) + 127;
}

// 1 / X of a block's code, X = 2^(code - 127), as a float: exact for the
// codes of finite float blocks (at most 246); 1 for the NaN code, whose
// element codes are replaced by kMxNanCodes anyway.
__device__ __forceinline__ float mx_inv_scale(int code) {
  return __uint_as_float(static_cast<uint32_t>(code == kMxNanScale ? 127 : 254 - code) << 23);
}

// E4M3 codes of a * inv .. d * inv (round to nearest even, saturating at
// +-448), a in the low byte. v * 2^-s is exact (a power-of-two scaling that
// stays in the normal range for every value that can round to a non-zero
// E4M3), so the E4M3 conversion is the only rounding.
__device__ __forceinline__ uint32_t mx_encode4(float a, float b, float c, float d, float inv) {
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(a * inv, b * inv), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(c * inv, d * inv), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// One block of 32 values, given as floats v and as the same values packed in
// bf16 pairs (v2, for the block maximum): returns the E8M0 code of its scale
// and packs the 32 E4M3 codes four to a word (element 4i in the low byte of
// word i).
__device__ __forceinline__ uint8_t quantize_block32(const float* v, const uint32_t* v2,
                                                    uint32_t* words) {
  const int code = mx_block_code(bf16x2_absmax_bits<16>(v2));
  const float inv = mx_inv_scale(code);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = mx_encode4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], inv);
    words[i] = code == kMxNanScale ? kMxNanCodes : w;
  }
  return static_cast<uint8_t>(code);
}

// Tiled scale layout read by the block-scaled MMA. Scales of a [rows, K]
// operand (rows % 128 == 0, K % 128 == 0) are grouped by 128-row block rb
// and 128-wide K group kg into 512-byte atoms, atom (rb, kg) at
// (rb * (K / 128) + kg) * 512; inside an atom the scale of row m
// (0 <= m < 128) for 32-block kk (0..3) of the group sits at byte
// (m % 32) * 16 + (m / 32) * 4 + kk. An atom is what one
// tcgen05.cp.32x128b.warpx4 moves into tensor memory.
__host__ __device__ __forceinline__ int64_t mx_scale_offset(int64_t row, int64_t kblock32,
                                                            int64_t K) {
  const int64_t rb = row >> 7, m = row & 127;
  const int64_t kg = kblock32 >> 2, kk = kblock32 & 3;
  return (rb * (K >> 7) + kg) * 512 + (m & 31) * 16 + (m >> 5) * 4 + kk;
}

}  // namespace moe
