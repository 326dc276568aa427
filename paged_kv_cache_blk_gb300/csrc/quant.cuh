// Quantisation of one token row's heads for int8 pools, shared by the
// quantising scatter (copy_kernels.cu) and the fused decode step
// (decode.cu), so both store the same bytes.
//
// One warp per (token, kv head), VPL = head_dim / 32 values per lane:
// absmax of the head (fp32, a warp max over the |x| bit patterns), scale =
// absmax / 127 and code = round_half_even(x / scale), both divisions IEEE
// fp32 with subnormals kept (div.rn.f32 without .ftz, whatever the fast-math
// flags), codes clamped to [-127, 127].  A zero absmax stores scale 0 and
// codes 0.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace pkv {

__device__ __forceinline__ float div_ieee(float a, float b) {
  float r;
  asm("div.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

template <int VPL>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* src, float (&x)[VPL]) {
  if constexpr (VPL == 8) {
    const uint4 r = *reinterpret_cast<const uint4*>(src);
    x[0] = bf16_lo(r.x); x[1] = bf16_hi(r.x); x[2] = bf16_lo(r.y); x[3] = bf16_hi(r.y);
    x[4] = bf16_lo(r.z); x[5] = bf16_hi(r.z); x[6] = bf16_lo(r.w); x[7] = bf16_hi(r.w);
  } else if constexpr (VPL == 4) {
    const uint2 r = *reinterpret_cast<const uint2*>(src);
    x[0] = bf16_lo(r.x); x[1] = bf16_hi(r.x); x[2] = bf16_lo(r.y); x[3] = bf16_hi(r.y);
  } else if constexpr (VPL == 2) {
    const uint32_t r = *reinterpret_cast<const uint32_t*>(src);
    x[0] = bf16_lo(r); x[1] = bf16_hi(r);
  } else {
    x[0] = __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(src)) << 16);
  }
}

// Quantise one head (VPL values per lane); returns the scale, codes in c.
template <int VPL>
__device__ __forceinline__ float quantise_head(const float (&x)[VPL], int (&c)[VPL]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) m = max(m, __float_as_uint(x[i]) & 0x7FFFFFFFu);
  m = __reduce_max_sync(0xffffffffu, m);
  const float scale = div_ieee(__uint_as_float(m), 127.f);
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    c[i] = m == 0 ? 0 : min(127, max(-127, __float2int_rn(div_ieee(x[i], scale))));
  return scale;
}

// Codes are stored offset binary: the byte of code c is c + 128.
template <int VPL>
__device__ __forceinline__ void store_codes(char* dst, const int (&c)[VPL]) {
  uint32_t w[(VPL + 3) / 4] = {};
#pragma unroll
  for (int i = 0; i < VPL; ++i) w[i / 4] |= (uint32_t)((c[i] + 128) & 0xFF) << (8 * (i % 4));
  if constexpr (VPL == 8) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  } else if constexpr (VPL == 4) {
    *reinterpret_cast<uint32_t*>(dst) = w[0];
  } else if constexpr (VPL == 2) {
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w[0];
  } else {
    *reinterpret_cast<uint8_t*>(dst) = (uint8_t)w[0];
  }
}

}  // namespace pkv
