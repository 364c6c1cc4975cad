// nvfp4.cuh -- NVFP4 weight decoding for the W4A16 GEMMs (flashinfer PR #4048: NVFP4 weights,
// BF16 activations; E2M1 codes with one E4M3 scale per 16 consecutive k, and an FP32 per-expert
// scale that the epilogue applies to the FP32 accumulator).
//
// A decoded weight must be the exact bf16 value of e2m1 * e4m3 (both have few enough mantissa
// bits that the product always is one).  The hardware converts E2M1 pairs only to f16x2
// (cvt.rn.f16x2.e2m1x2), so each f16 half is moved into bf16 position by shifting its exponent
// and mantissa right by 3 bits with the sign kept: the bf16 read from those bits is the f16
// value times 2^-112 (f16 bias 15 against bf16 bias 127).  Every E2M1 value is a normal f16, so
// this is exact, and zero stays zero.  The block scale is carried as bf16(e4m3 * 2^112), exact
// and below the bf16 maximum (448 * 2^112 < 2^121), so one bf16x2 multiply restores the value
// and applies the scale in the same exact step.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gb300moe {

// Four E4M3 block scales (bytes of `sf4`, lowest first) -> bf16x2 words holding
// scale * 2^112 in both halves.
__device__ __forceinline__ void nvfp4_scales(uint32_t sf4, uint32_t (&s2)[4]) {
  uint32_t h01, h23;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}\n"
      : "=r"(h01), "=r"(h23)
      : "r"(sf4));
  const float f[4] = {__half2float(__ushort_as_half((unsigned short)(h01 & 0xFFFFu))),
                      __half2float(__ushort_as_half((unsigned short)(h01 >> 16))),
                      __half2float(__ushort_as_half((unsigned short)(h23 & 0xFFFFu))),
                      __half2float(__ushort_as_half((unsigned short)(h23 >> 16)))};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float v = f[i] * 0x1p112f;  // exact: a power-of-two scaling of an f32 value
    const __nv_bfloat162 b = __floats2bfloat162_rn(v, v);
    s2[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// Eight E2M1 codes (two per byte of `w`, element 2i in the low nibble) times one block scale
// word from nvfp4_scales -> four bf16x2 words, elements in order (low half first).
__device__ __forceinline__ void nvfp4_decode8(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}\n"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t y = ((h[i] & 0x7FFF7FFFu) >> 3) | (h[i] & 0x80008000u);
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(y), "r"(s2));
  }
}

}  // namespace gb300moe
