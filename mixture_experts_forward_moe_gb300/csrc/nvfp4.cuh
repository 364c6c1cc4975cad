// nvfp4.cuh -- NVFP4 weight decoding for the W4A16 GEMMs (flashinfer PR #4048: NVFP4 weights,
// 16-bit activations; E2M1 codes with one E4M3 scale per 16 consecutive k, and an FP32
// per-expert scale that the epilogue applies to the FP32 accumulator).
//
// The decoded weight is the exact f16 value of e2m1 * e4m3, and the NVFP4 GEMMs multiply it
// with f16 tokens.  Both factors convert to f16 exactly (E2M1: 0, 0.5 .. 6; E4M3: 2^-9 .. 448,
// all f16 normals), and so does their product: at most six significant bits, magnitude 0 or
// between 2^-10 and 6 * 448 = 2688.  The hardware converts E2M1 and E4M3 pairs to f16x2 in one
// instruction each, so a pair of weights costs a conversion and one f16x2 multiply (a decode to
// bf16 needs a bit shift and a rebias on top, about two and a half times the instructions).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gb300moe {

// Four E4M3 block scales (bytes of `sf4`, lowest first) -> f16x2 words holding one scale in
// both halves.
__device__ __forceinline__ void nvfp4_scales(uint32_t sf4, uint32_t (&s2)[4]) {
  uint32_t h01, h23;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}\n"
      : "=r"(h01), "=r"(h23)
      : "r"(sf4));
  s2[0] = __byte_perm(h01, h01, 0x1010);
  s2[1] = __byte_perm(h01, h01, 0x3232);
  s2[2] = __byte_perm(h23, h23, 0x1010);
  s2[3] = __byte_perm(h23, h23, 0x3232);
}

// Eight E2M1 codes (two per byte of `w`, element 2i in the low nibble) times one block scale
// word from nvfp4_scales -> four f16x2 words, elements in order (low half first).
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
  for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(h[i]), "r"(s2));
}

}  // namespace gb300moe
