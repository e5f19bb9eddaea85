// mx.cuh -- MXFP8 helpers shared by the MXFP8 kernels: the blocked scale-tile
// layout, e4m3 packing and the per-32 requantization of the activation.
//
// Scale tiles ("Prime Flash MoE" sec. 7 "Scales are piped through tensor
// memory"; "Porting Block-Scaled GEMM Kernels" sec. 1.2: 512-byte chunks of
// 128 rows x 4 K-scales): the scales of rows [128 rt, 128 rt + 128) and K
// columns [128 kt, 128 kt + 128) form one 512-byte tile at
//     (rt * (K/128) + kt) * 512,
// with the scale of tile row r and 32-column group g at byte
//     (r % 32) * 16 + (r / 32) * 4 + g
// -- 32 rows of 16 bytes, the shape tcgen05.cp .32x128b.warpx4 copies into
// four TMEM columns (one per group of 32 rows, one byte per K group).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace moe {

__host__ __device__ __forceinline__ int64_t sf_tile_offset(int64_t row_tile, int k_tile, int k_tiles) {
  return (row_tile * k_tiles + k_tile) * 512;
}
__host__ __device__ __forceinline__ int sf_in_tile(int r) { return ((r & 31) << 4) + ((r >> 5) << 2); }

// Two floats -> two e4m3 codes (round to nearest even, saturating to +-448),
// `lo` in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Requantize 32 fp32 values to MXFP8 (sec. 7 "The epilogue also quantizes"):
// scale exponent e = ceil(log2(amax / 448)), the smallest e with
// amax * 2^-e <= 448 ("Porting Block-Scaled GEMM Kernels" sec. 6.2: the scale
// is amax/448 rounded up to a power of two), computed exactly from the bits of
// amax = m 2^p (m in [1,2)): e = p - 8 + (m > 1.75).  amax == 0 gives e = 0.
// Writes the 32 codes into q[0..7] (little-endian bytes) and returns the
// e8m0 scale byte e + 127.
__device__ __forceinline__ uint32_t mx_quantize32(const float* a, uint32_t (&q)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(a[i]));
  const uint32_t bits = __float_as_uint(amax);
  int e = 0;
  if (amax > 0.f) {
    const int p = (int)((bits >> 23) & 0xff) - 127;
    e = p - 8 + ((bits & 0x7fffff) > 0x600000u ? 1 : 0);
    e = max(e, -127);
  }
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e exactly
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = cvt_e4m3x2(a[4 * i] * inv, a[4 * i + 1] * inv);
    const uint32_t hi = cvt_e4m3x2(a[4 * i + 2] * inv, a[4 * i + 3] * inv);
    q[i] = lo | (hi << 16);
  }
  return (uint32_t)(e + 127);
}

// Shared-memory descriptor of one 512-byte scale tile for tcgen05.cp: no
// swizzle, 8-row x 16-byte core matrices, 128 bytes between them.
__device__ __forceinline__ uint64_t sdesc_sf_tile(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(128u >> 4) << 32) |
         ((uint64_t)1u << 46);
}

// TMEM <- 512-byte scale tile (32 lanes x 128 bits, replicated to the four
// lane quadrants).
__device__ __forceinline__ void utccp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D (+)= (A * sfA) (B * sfB)^T, e4m3 operands with one ue8m0 scale per 32
// along K (kind::mxf8f6f4, block_scale, scale_vec::1X).
__device__ __forceinline__ void umma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Instruction descriptor of the block-scaled kinds ("Porting Block-Scaled
// GEMM Kernels" sec. 1.3 lists the fields): A and B e4m3 (format code 0 under
// kind::mxf8f6f4, sec. 2.3), both K-major, N>>3 at bits 17-22, scale type
// UE8M0 at bit 23, M>>7 at bits 27-28.  The scale selectors (bits 29-30 for
// A, 4-5 for B) pick the byte of each 32-bit scale word: the K group.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 7) << 27);
}
// Format code of E2M1 (FP4) for an operand of kind::mxf8f6f4 (bits 7-9 for A,
// 10-12 for B; "Porting Block-Scaled GEMM Kernels" sec. 2.3: 5 under this
// kind, while 1 would read as E5M2).
constexpr uint32_t kFmtE2M1 = 5;
__device__ __forceinline__ uint32_t idesc_with_sf_id(uint32_t idesc, uint32_t k_group) {
  return idesc | (k_group << 29) | (k_group << 4);
}

// global -> shared bulk copy completing on an mbarrier (16-byte granular).
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(sdst)),
               "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

}  // namespace moe
