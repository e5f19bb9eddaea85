// mx4.cu -- MXFP4 expert weights (E2M1 codes, two per byte, one ue8m0 scale
// per 32 elements: the routed-weight format of "GC-MoE on SM120" sec. 2.2)
// widened to e4m3 codes, so that the block-scaled MXFP8 GEMMs run them with
// the same scales.  Every E2M1 value is an e4m3 value, so the widening is
// exact and the products equal those of the 4-bit operands.
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {
namespace {

// e4m3 codes of the eight E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, as the
// eight bytes of two words (selector i picks byte i)
constexpr uint32_t kMagLo = 0x3C383000u;  // 0x00 0x30 0x38 0x3C
constexpr uint32_t kMagHi = 0x4C484440u;  // 0x40 0x44 0x48 0x4C

// Four E2M1 codes (the low 16 bits of w, element i in bits 4i..4i+3) to four
// e4m3 bytes (element i in byte i).
__device__ __forceinline__ uint32_t widen4(uint32_t w) {
  const uint32_t mag = __byte_perm(kMagLo, kMagHi, w & 0x7777u);
  const uint32_t s = w & 0x8888u;  // sign bit 4i+3 -> bit 8i+7
  const uint32_t sign = ((s & 0x8u) << 4) | ((s & 0x80u) << 8) | ((s & 0x800u) << 12) | ((s & 0x8000u) << 16);
  return mag | sign;
}

// Grid-stride over 16-byte chunks of the packed input: each chunk (32
// elements) becomes two 16-byte chunks of codes.
__global__ void __launch_bounds__(256) widen_e2m1_kernel(const uint4* __restrict__ in, int64_t n16,
                                                         uint4* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 v = __ldg(in + i);
    uint4 a, b;
    a.x = widen4(v.x);
    a.y = widen4(v.x >> 16);
    a.z = widen4(v.y);
    a.w = widen4(v.y >> 16);
    b.x = widen4(v.z);
    b.y = widen4(v.z >> 16);
    b.z = widen4(v.w);
    b.w = widen4(v.w >> 16);
    out[2 * i] = a;
    out[2 * i + 1] = b;
  }
}

}  // namespace

// n_bytes: packed input bytes, a multiple of 16; out holds 2 * n_bytes.
cudaError_t launch_widen_e2m1(const void* in, int64_t n_bytes, void* out, int grid, cudaStream_t stream) {
  const int64_t n16 = n_bytes / 16;
  const int64_t need = (n16 + 255) / 256;
  const int g = (int)(need < grid ? need : grid);
  if (g <= 0) return cudaSuccess;
  widen_e2m1_kernel<<<g, 256, 0, stream>>>(static_cast<const uint4*>(in), n16, static_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace moe
