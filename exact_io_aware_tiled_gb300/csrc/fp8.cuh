// fp8.cuh -- device helpers of the FP8 (E4M3) forward path (sm_103a).
//
//   * E4M3 conversion (cvt.rn.satfinite: round to nearest even, saturating
//     at +-448, the format's largest finite value);
//   * the fast Walsh-Hadamard transform of a register-resident row, in a
//     fixed butterfly order (stage h = 1, 2, ..., D/2 pairs i and i + h) so
//     that every implementation of the same order gets the same float32
//     bits;
//   * the 64-byte-swizzle shared-memory descriptor and tcgen05.mma
//     kind::f8f6f4 (both operands E4M3 from shared memory, float32
//     accumulation in tensor memory).
#pragma once
#include "common.cuh"

namespace fa {

// Packs E4M3(lo) into bits 0-7 and E4M3(hi) into bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Four E4M3 bytes, x0 in bits 0-7.
__device__ __forceinline__ uint32_t e4m3x4(float x0, float x1, float x2, float x3) {
  return e4m3x2(x0, x1) | (e4m3x2(x2, x3) << 16);
}

// x <- x H_D (Sylvester order), in place, float32 adds and subtracts.  From
// stage h = 2 on, the butterflies of i and i + 1 (both with bit h clear) run
// as one packed f32x2 add and one packed subtract; each lane rounds exactly
// as the scalar operation would, so the result is bit for bit the same.
template <int D>
__device__ __forceinline__ void fwht_rows(float (&x)[D]) {
#pragma unroll
  for (int i = 0; i < D; i += 2) {
    const float a = x[i], b = x[i + 1];
    x[i] = __fadd_rn(a, b);
    x[i + 1] = __fsub_rn(a, b);
  }
#pragma unroll
  for (int h = 2; h < D; h <<= 1) {
#pragma unroll
    for (int i = 0; i < D; i += 2) {
      if ((i & h) == 0) {
        float s0 = x[i], s1 = x[i + 1], d0, d1;
        sub2(d0, d1, s0, s1, x[i + h], x[i + h + 1]);
        add2(s0, s1, x[i + h], x[i + h + 1]);
        x[i] = s0;
        x[i + 1] = s1;
        x[i + h] = d0;
        x[i + h + 1] = d1;
      }
    }
  }
}

// x[c] <- x[c] * k, packed in pairs (one rounding per lane, as scalar).
template <int D>
__device__ __forceinline__ void scale_rows(float (&x)[D], float k) {
#pragma unroll
  for (int c = 0; c < D; c += 2) mul2(x[c], x[c + 1], x[c], x[c + 1], k, k);
}

// Shared-memory matrix descriptor, 64-byte swizzle (swizzle mode 4 in bits
// 61-63 of the sm_100 family format): K-major rows of 64 bytes, 8-row
// groups 512 bytes apart.  Tiles are 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;
  return d;
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A and B (format 0),
// float32 accumulation, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], E4M3 operands (K = 32 per instruction).
__device__ __forceinline__ void mma_ss_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

}  // namespace fa
