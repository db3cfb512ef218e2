// Device helpers shared by the NVFP4 kernels: exact E2M1 / E4M3 decode into
// packed half registers, and small load/store wrappers.
//
// Format (mlxcel issue #693 "direct-transcode ModelOpt triplets to MLX
// native", Technical notes): a uint32 word holds eight E2M1 codes, column
// 8*j+i in nibble i (least significant first); one E4M3 byte scales each run
// of 16 columns. E2M1 magnitudes are 0, .5, 1, 1.5, 2, 3, 4, 6; bit 3 is the
// sign. The product fp4 * e4m3 has at most 6 significant bits and lies in
// [2^-10, 2688], so it is exact in f16, bf16 and f32; every decode below is
// exact.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nvfp4 {

// 448 * 6: the global scale enters as gs / 2688 once per output (mlxcel PR
// #2629, Summary).
constexpr float kGlobalScaleDivisor = 2688.0f;

__device__ __forceinline__ float global_factor(const float* gs, int64_t e) {
  return gs ? __fdiv_rn(__ldg(gs + e), kGlobalScaleDivisor) : 1.0f;
}

// Four E2M1 nibble pairs (the bytes of w) -> four f16x2 registers. Byte b
// gives register b: low nibble in the low half, high nibble in the high half.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2. E4M3 fits f16 exactly
// (largest 448, smallest subnormal 2^-9); NaN bytes give NaN.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)(two_bytes & 0xFFFFu)));
  return r;
}

// One E4M3 byte broadcast into both halves of an f16x2.
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t byte) {
  return e4m3x2_to_f16x2((byte & 0xFFu) * 0x0101u);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  const uint32_t h = e4m3x2_to_f16x2(byte & 0xFFu);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// E4M3 byte -> bf16x2 broadcast of scale * 2^112 (exact: a 4-bit significand
// and |scale * 2^112| <= 448 * 2^112 < 2^121 fit bf16).
__device__ __forceinline__ uint32_t e4m3_to_bf16x2_bcast_x2p112(uint32_t byte) {
  const float s = e4m3_to_f32(byte) * 0x1p112f;
  const __nv_bfloat16 b = __float2bfloat16_rn(s);
  const uint32_t u = __bfloat16_as_ushort(b);
  return u | (u << 16);
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Eight E2M1 codes times one block scale -> four packed f16x2 (exact).
// sc = e4m3_to_f16x2_bcast(scale byte).
__device__ __forceinline__ void decode8_scaled_f16(uint32_t w, uint32_t sc, uint32_t (&out)[4]) {
  uint32_t h[4];
  e2m1x8_to_f16x2(w, h);
#pragma unroll
  for (int b = 0; b < 4; ++b) out[b] = hmul2_f16(h[b], sc);
}

// Eight E2M1 codes times one block scale -> four packed bf16x2 (exact).
// sc = e4m3_to_bf16x2_bcast_x2p112(scale byte).
//
// There is no E2M1 -> bf16 conversion instruction, so the magnitudes are
// decoded to f16 first. An f16 E2M1 magnitude has zero low mantissa bits, so
// shifting its bit pattern right by three gives the bf16 pattern of
// value * 2^-112 (same exponent field, shorter mantissa) without disturbing
// the neighbouring half. The nibble sign bits are moved to bits 15 and 31 by
// one byte permute, and the single bf16 multiply by scale * 2^112 restores the
// exact product fp4 * scale.
__device__ __forceinline__ void decode8_scaled_bf16(uint32_t w, uint32_t sc, uint32_t (&out)[4]) {
  uint32_t h[4];
  e2m1x8_to_f16x2(w & 0x77777777u, h);
  const uint32_t w4 = w << 4;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    // byte 1 <- byte b of (w << 4): its bit 7 is the low nibble's sign.
    // byte 3 <- byte b of w: its bit 7 is the high nibble's sign.
    const uint32_t sg = __byte_perm(w4, w, (uint32_t)((b << 4) | ((4 + b) << 12)));
    const uint32_t mag = h[b] >> 3;
    out[b] = hmul2_bf16(mag | (sg & 0x80008000u), sc);
  }
}

template <typename T> struct Dt;
template <> struct Dt<__half> {
  __device__ static __forceinline__ uint32_t scale(uint32_t byte) { return e4m3_to_f16x2_bcast(byte); }
  __device__ static __forceinline__ void decode(uint32_t w, uint32_t sc, uint32_t (&o)[4]) { decode8_scaled_f16(w, sc, o); }
  __device__ static __forceinline__ __half from_f32(float v) { return __float2half_rn(v); }
};
template <> struct Dt<__nv_bfloat16> {
  __device__ static __forceinline__ uint32_t scale(uint32_t byte) { return e4m3_to_bf16x2_bcast_x2p112(byte); }
  __device__ static __forceinline__ void decode(uint32_t w, uint32_t sc, uint32_t (&o)[4]) { decode8_scaled_bf16(w, sc, o); }
  __device__ static __forceinline__ __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Streaming (evict-first) 128-bit load for data read once per call.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.cs.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

}  // namespace nvfp4
