// Bandwidth-bound kernels: ModelOpt-triplet transcode and exact dequantize.
#include <cstdlib>

#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_pipe.cuh"

namespace nvfp4 {

__device__ int g_copy_error = 0;  // first error code recorded by a bounded wait of the bulk copy

namespace {

constexpr int kStreamThreads = 256;

// Grid for a grid-stride kernel: enough blocks for `units` thread-iterations,
// at most what is resident at once (a second wave of equal blocks would run
// after the first instead of beside it).
template <typename Kern>
int stream_grid(Kern kern, int64_t units) {
  int dev = 0, sms = 152, per_sm = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStreamThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t want = (units + kStreamThreads - 1) / kStreamThreads;
  const int64_t cap = (int64_t)sms * per_sm;
  return (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

// Transcode (issue #693 "direct-transcode ModelOpt triplets to MLX native",
// Implementation plan step 3). ModelOpt's U8 plane stores column 2j in the
// low nibble of byte j; packing four consecutive bytes little-endian into one
// uint32 therefore yields the native word with column 8i+k in nibble k. That
// repack is the identity on the byte stream, so the kernel copies both planes
// as they are; the E4M3 block scales are kept byte for byte and the sidecar is
// f32(ws2) * 2688 so that gs / 2688 stands for ws2. Both planes are read and
// written exactly once; no dense intermediate.
//
// The copy engine moves the bytes: each CTA (one per SM, one thread issuing)
// copies a contiguous run of 32 KB chunks of both planes through a ring of
// six shared-memory buffers, bulk loads running up to six chunks ahead of the
// bulk stores, a handful of instructions per 32 KB (a 16-byte vector copy
// with eight loads in flight per thread took 80 us for a layer's three
// triplets, this one 75). Sizes and addresses of bulk copies must be
// multiples of 16 bytes: the last (< 16) bytes of each plane are copied by
// plain stores.
constexpr uint32_t kCopyChunk = 32 * 1024;
constexpr int kCopyBufs = 6;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(32, 1)
transcode_bulk_kernel(const uint8_t* __restrict__ mo_w, int64_t w_bytes, const uint8_t* __restrict__ mo_ws,
                      int64_t s_bytes, const float* __restrict__ ws2, uint8_t* __restrict__ w_out,
                      uint8_t* __restrict__ s_out, float* __restrict__ gs_out) {
  extern __shared__ __align__(128) uint8_t buf[];
  __shared__ __align__(8) uint64_t bars[kCopyBufs];
  __shared__ int abort_flag;
  const int64_t wv = w_bytes & ~(int64_t)15, sv = s_bytes & ~(int64_t)15;
  const int64_t n0 = (wv + kCopyChunk - 1) / kCopyChunk, n = n0 + (sv + kCopyChunk - 1) / kCopyChunk;
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) gs_out[0] = __fmul_rn(__ldg(ws2), kGlobalScaleDivisor);
    if (threadIdx.x < w_bytes - wv) w_out[wv + threadIdx.x] = mo_w[wv + threadIdx.x];
    if (threadIdx.x < s_bytes - sv) s_out[sv + threadIdx.x] = mo_ws[sv + threadIdx.x];
  }
  if (threadIdx.x != 0) return;
  // chunk c: source, destination and size
  auto chunk = [&](int64_t c, const uint8_t*& src, uint8_t*& dst, uint32_t& bytes) {
    if (c < n0) {
      const int64_t off = c * kCopyChunk;
      src = mo_w + off;
      dst = w_out + off;
      bytes = (uint32_t)(wv - off < kCopyChunk ? wv - off : kCopyChunk);
    } else {
      const int64_t off = (c - n0) * kCopyChunk;
      src = mo_ws + off;
      dst = s_out + off;
      bytes = (uint32_t)(sv - off < kCopyChunk ? sv - off : kCopyChunk);
    }
  };
  const int64_t c0 = n * blockIdx.x / gridDim.x, c1 = n * (blockIdx.x + 1) / gridDim.x;
  const uint32_t sbuf = pipe::smem_addr(buf), sbar = pipe::smem_addr(bars);
  abort_flag = 0;
  for (int k = 0; k < kCopyBufs; ++k) pipe::mbar_init(sbar + 8u * k, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  int64_t issued = c0;  // next chunk to load
  for (; issued < c1 && issued < c0 + kCopyBufs; ++issued) {
    const uint8_t* src;
    uint8_t* dst;
    uint32_t bytes;
    chunk(issued, src, dst, bytes);
    const int k = (int)(issued - c0);
    pipe::mbar_arrive_tx(sbar + 8u * k, bytes);
    bulk_g2s(sbuf + (uint32_t)k * kCopyChunk, src, bytes, sbar + 8u * k);
  }
  int64_t i = c0;
  for (; i < c1; ++i) {
    const int k = (int)((i - c0) % kCopyBufs);
    const uint32_t ph = (uint32_t)(((i - c0) / kCopyBufs) & 1);
    if (!pipe::wait_bar(sbar + 8u * k, ph, &abort_flag, 41, &g_copy_error)) break;
    const uint8_t* src;
    uint8_t* dst;
    uint32_t bytes;
    chunk(i, src, dst, bytes);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bulk_s2g(dst, sbuf + (uint32_t)k * kCopyChunk, bytes);
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    if (issued < c1) {
      // buffer k is reloaded once the store just issued has read it
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      chunk(issued, src, dst, bytes);
      pipe::mbar_arrive_tx(sbar + 8u * k, bytes);
      bulk_g2s(sbuf + (uint32_t)k * kCopyChunk, src, bytes, sbar + 8u * k);
      ++issued;
    }
  }
  // No load may still be in flight into shared memory when the CTA exits
  // (only after a wait gave up), and the stores must have completed.
  for (int64_t v = i; v < issued; ++v)
    pipe::wait_bar_quiet(sbar + 8u * (uint32_t)((v - c0) % kCopyBufs), (uint32_t)(((v - c0) / kCopyBufs) & 1));
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Exact dequantize (PR #2629 "ROCm native NVFP4", Summary: the dequantize
// kernel expands a plane exactly; Changes during review: the grid is sized
// from the weight plane). One thread-iteration expands one packed word (half
// of a 16-column block): eight outputs from the word and its block's scale
// byte, so that a warp's output store is 32 x 16 contiguous bytes (bf16/f16).
// Element value = cast(f32(fp4 * e4m3) * factor) with factor = gs[e] / 2688
// (absent gs: the product itself, exact in every output type).
template <typename OutT>
__device__ __forceinline__ void store8(OutT* dst, const uint32_t (&h)[4], float fac, bool has_gs);

__device__ __forceinline__ float h_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFF))); }
__device__ __forceinline__ float h_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

template <>
__device__ __forceinline__ void store8<float>(float* dst, const uint32_t (&h)[4], float fac, bool has_gs) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = h_lo(h[i]);
    v[2 * i + 1] = h_hi(h[i]);
  }
  if (has_gs) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], fac);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 2; ++q)
    __stcs(d + q, make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                             __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3])));
}

template <>
__device__ __forceinline__ void store8<__half>(__half* dst, const uint32_t (&h)[4], float fac, bool has_gs) {
  uint32_t o[4];
  if (!has_gs) {
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = h[i];
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half lo = __float2half_rn(__fmul_rn(h_lo(h[i]), fac));
      const __half hi = __float2half_rn(__fmul_rn(h_hi(h[i]), fac));
      o[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
  }
  __stcs(reinterpret_cast<uint4*>(dst), make_uint4(o[0], o[1], o[2], o[3]));
}

template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const uint32_t (&h)[4], float fac,
                                                      bool has_gs) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = h_lo(h[i]), b = h_hi(h[i]);
    if (has_gs) {
      a = __fmul_rn(a, fac);
      b = __fmul_rn(b, fac);
    }
    o[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
  }
  __stcs(reinterpret_cast<uint4*>(dst), make_uint4(o[0], o[1], o[2], o[3]));
}

template <typename OutT>
__global__ void __launch_bounds__(kStreamThreads)
dequantize_kernel(const uint32_t* __restrict__ w, const uint8_t* __restrict__ scales,
                  const float* __restrict__ gs, int64_t E, int64_t words_per_expert,
                  OutT* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = blockIdx.y; e < E; e += gridDim.y) {
    const float fac = global_factor(gs, e);
    const bool has_gs = gs != nullptr;
    const int64_t base = e * words_per_expert;  // first word of expert e
    // kU words per thread and iteration, all loads issued before any decode
    // so that their latencies overlap.
    constexpr int kU = 8;
    int64_t vi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; vi + (kU - 1) * stride < words_per_expert; vi += kU * stride) {
      uint32_t wv[kU], sb[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t v = base + vi + u * stride;
        wv[u] = __ldcs(w + v);
        sb[u] = __ldcs(scales + (v >> 1));
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t v = base + vi + u * stride;
        uint32_t h[4];
        decode8_scaled_f16(wv[u], e4m3_to_f16x2_bcast(sb[u]), h);
        store8<OutT>(out + 8 * v, h, fac, has_gs);
      }
    }
    for (; vi < words_per_expert; vi += stride) {
      const int64_t v = base + vi;
      uint32_t h[4];
      decode8_scaled_f16(__ldcs(w + v), e4m3_to_f16x2_bcast(__ldcs(scales + (v >> 1))), h);
      store8<OutT>(out + 8 * v, h, fac, has_gs);
    }
  }
}

// ---------------------------------------------------------------- quantize
//
// Dense -> NVFP4 (the encoding half of MLX's global-scale convention, mlx PR
// #2629, Implementation Review Summary: block scales are encoded times
// 448 * 6 / global_scale). Per 16-column block, in IEEE float32:
// amax = max |x|, s = amax / 6 (times 2688 / gs with a global scale), scale
// byte = E4M3 nearest to s (ties to even, saturating at 448), d = e4m3 * gs /
// 2688, r = 1 / d, code = E2M1 nearest to x * r (ties to even, saturating at
// +-6), +0 for a zero magnitude, all codes 0 where d == 0. Both roundings are
// the hardware conversions (cvt.rn.satfinite); one reciprocal per block
// instead of a division per element keeps the kernel bound by HBM.

__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float v) {
  unsigned short h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(v));
  return (uint32_t)h & 0xFFu;
}

// One 16-column block's inputs as raw 16-byte words (four for f32).
template <typename T> struct Raw16 { uint4 q[sizeof(T) == 4 ? 4 : 2]; };

__device__ __forceinline__ uint32_t u4get(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// max |x| over a block. For 16-bit inputs the maximum is taken on the packed
// halves: max.xorsign.abs gives max(|a|, |b|) (exact) with some sign, which
// the next step ignores and the end clears; one widening at the end.
template <typename T> __device__ __forceinline__ float amax16(const Raw16<T>& r);
template <> __device__ __forceinline__ float amax16<float>(const Raw16<float>& r) {
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(__uint_as_float(u4get(r.q[i >> 2], i & 3))));
  return am;
}
template <> __device__ __forceinline__ float amax16<__nv_bfloat16>(const Raw16<__nv_bfloat16>& r) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(u4get(r.q[i >> 2], i & 3)));
  m &= 0x7FFF7FFFu;
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}
template <> __device__ __forceinline__ float amax16<__half>(const Raw16<__half>& r) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) asm("max.xorsign.abs.f16x2 %0, %0, %1;" : "+r"(m) : "r"(u4get(r.q[i >> 2], i & 3)));
  m &= 0x7FFF7FFFu;
  return fmaxf(__half2float(__ushort_as_half((unsigned short)(m & 0xFFFFu))),
               __half2float(__ushort_as_half((unsigned short)(m >> 16))));
}

// Columns 2i and 2i + 1 of a block as f32 (i = 0..7).
template <typename T> __device__ __forceinline__ void pair_at(const Raw16<T>& r, int i, float& lo, float& hi);
template <> __device__ __forceinline__ void pair_at<float>(const Raw16<float>& r, int i, float& lo, float& hi) {
  lo = __uint_as_float(u4get(r.q[i >> 1], 2 * (i & 1)));
  hi = __uint_as_float(u4get(r.q[i >> 1], 2 * (i & 1) + 1));
}
template <> __device__ __forceinline__ void pair_at<__nv_bfloat16>(const Raw16<__nv_bfloat16>& r, int i, float& lo,
                                                                 float& hi) {
  const uint32_t u = u4get(r.q[i >> 2], i & 3);
  lo = __uint_as_float(u << 16);
  hi = __uint_as_float(u & 0xFFFF0000u);
}
template <> __device__ __forceinline__ void pair_at<__half>(const Raw16<__half>& r, int i, float& lo, float& hi) {
  const uint32_t u = u4get(r.q[i >> 2], i & 3);
  lo = __half2float(__ushort_as_half((unsigned short)(u & 0xFFFFu)));
  hi = __half2float(__ushort_as_half((unsigned short)(u >> 16)));
}

// (a, b) * (r, r), each product rounded to nearest (one packed multiply).
__device__ __forceinline__ void mul2_rn(float& a, float& b, float r) {
  uint64_t p, q, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(q) : "f"(r));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(p), "l"(q));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
}

// Four (low, high) pairs -> one word of eight E2M1 codes, low column in the
// low nibble (cvt puts its first source in the high nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* lo, const float* hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(lo[0]), "f"(hi[0]), "f"(lo[1]), "f"(hi[1]), "f"(lo[2]), "f"(hi[2]), "f"(lo[3]), "f"(hi[3]));
  return r;
}
// +0 for every zero magnitude (a negative value that rounds to zero): a
// nibble keeps its sign bit only where its magnitude m is nonzero, i.e.
// where m + 7 (at most 14: no carry between nibbles) reaches bit 3.
__device__ __forceinline__ uint32_t plus_zero(uint32_t r) {
  const uint32_t m = r & 0x77777777u;
  return m | (r & (m + 0x77777777u) & 0x88888888u);
}

// Magnitude code of the E2M1 value nearest to the exact quotient a / d, for
// a >= 0 and d in [1, 2) (both scaled by the same power of two, which leaves
// the quotient as it is): a is compared with each midpoint m of the grid
// times d. fmaf forms a - m * d with one rounding, and with d in [1, 2) and
// a near m * d no result is small enough to underflow, so its sign is the
// exact comparison; a tie (+0) goes to the even code (up at 0.75, 1.75 and
// 3.5, down at the others). A quotient past 5 saturates at code 7 (6.0); a
// NaN compares false everywhere and gives 0.
__device__ __forceinline__ uint32_t e2m1_code_exact(float a, float d) {
  uint32_t c = 0;
  c += fmaf(-0.25f, d, a) > 0.0f;
  c += fmaf(-0.75f, d, a) >= 0.0f;
  c += fmaf(-1.25f, d, a) > 0.0f;
  c += fmaf(-1.75f, d, a) >= 0.0f;
  c += fmaf(-2.5f, d, a) > 0.0f;
  c += fmaf(-3.5f, d, a) >= 0.0f;
  c += fmaf(-5.0f, d, a) > 0.0f;
  return c;
}

// Element e of a block, read again from its copy in shared memory (at
// address blk) as float: the fix-up paths below are rare, and keeping the
// block's values in registers until then would cost registers everywhere.
template <typename T> __device__ __forceinline__ float elem_at(uint32_t blk, int e);
template <> __device__ __forceinline__ float elem_at<float>(uint32_t blk, int e) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(blk + 4u * (uint32_t)e));
  return v;
}
template <> __device__ __forceinline__ float elem_at<__nv_bfloat16>(uint32_t blk, int e) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(blk + 2u * (uint32_t)e));
  return __uint_as_float((uint32_t)v << 16);
}
template <> __device__ __forceinline__ float elem_at<__half>(uint32_t blk, int e) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(blk + 2u * (uint32_t)e));
  return __half2float(__ushort_as_half(v));
}

// Power-of-two scaling of a block's comparisons: |x| and d are multiplied by
// 2^-E, d = dn 2^E with dn in [1, 2), which leaves every quotient as it is.
// It is exact, except that an |x| far below d may lose bits (it stays below
// every midpoint) and one far above may become infinite (it stays above). A
// d below 2^-126 (a float32 subnormal) is first scaled by 2^126, and |x| with
// it, one power of two after the other.
struct Scaled {
  float pre, p, dn;
  __device__ __forceinline__ explicit Scaled(float d) {
    pre = d < 0x1p-126f ? 0x1p126f : 1.0f;
    const uint32_t db = __float_as_uint(d * pre);
    dn = __uint_as_float((db & 0x007FFFFFu) | 0x3F800000u);
    p = __uint_as_float((254u - (db >> 23)) << 23);  // 2^-E of d * pre, in [2^-125, 2^126]
  }
  __device__ __forceinline__ float operator()(float x) const { return (fabsf(x) * pre) * p; }
};

// The midpoint of E2M1 codes c and c + 1 (0.25, 0.75, 1.25, 1.75, 2.5, 3.5,
// 5 for c = 0..6): the float32 bits 0x3E800000 + (v << 21) with v = 0, 6, 9,
// 11, 13, 15, 17, byte c of a pair of 32-bit constants.
__device__ __forceinline__ float e2m1_midpoint(uint32_t c) {
  const uint32_t v = __byte_perm(0x0B090600u, 0x00110F0Du, c) & 0xFFu;
  return __uint_as_float(0x3E800000u + (v << 21));
}

// The values whose two conversions disagree (set nibbles of dm0 and dm1 for
// the words hw0 and hw1, elements 0..7 and 8..15 of the block; the codes in
// hw are those of the upper products). The products lie within a factor
// 1 + 2^-21 of each other and the midpoints at least a factor 1.4 apart, so
// exactly one midpoint m separates the two codes (c from the lower product,
// c + 1 from the upper one): the sign of |x| - m d picks one of them, and a
// tie the even one. fmaf forms |x| - m d with one rounding; for d >= 2^-100
// (callers send smaller d to exact_block) no nonzero result of it underflows
// to zero, so its sign is the exact comparison. Both words in one loop, so
// that a warp runs as many rounds as its lane with the most such values. The
// results still need plus_zero.
template <typename T>
__device__ __forceinline__ void fix_codes(uint32_t& hw0, uint32_t& hw1, uint32_t dm0, uint32_t dm1, uint32_t blk,
                                          float d) {
  while (dm0 | dm1) {
    const bool first = dm0 != 0;
    const uint32_t dm = first ? dm0 : dm1;
    const uint32_t hw = first ? hw0 : hw1;
    const int sh = (__ffs(dm) - 1) & ~3;
    const uint32_t nib = dm & (0xFu << sh);
    const uint32_t c = ((hw ^ nib) >> sh) & 7u;  // the lower product's code
    const float t = fmaf(-e2m1_midpoint(c), d, fabsf(elem_at<T>(blk, (first ? 0 : 8) + (sh >> 2))));
    const uint32_t flip = (t < 0.0f || (t == 0.0f && !(c & 1u))) ? nib : 0u;  // down to c
    if (first) {
      hw0 ^= flip;
      dm0 ^= nib;
    } else {
      hw1 ^= flip;
      dm1 ^= nib;
    }
  }
}

// Every code of a block by the full comparisons (a d whose reciprocal
// overflows float32). A zero magnitude gets +0.
template <typename T>
__device__ __forceinline__ uint2 exact_block(uint32_t blk, float d) {
  const Scaled sc(d);
  uint32_t wd[2] = {0u, 0u};
  for (int e = 0; e < 16; ++e) {
    const float x = elem_at<T>(blk, e);
    const uint32_t c = e2m1_code_exact(sc(x), sc.dn);
    const uint32_t nib = c | (c != 0u && x < 0.0f ? 8u : 0u);
    wd[e >> 3] |= nib << (4 * (e & 7));
  }
  return make_uint2(wd[0], wd[1]);
}

// One 16-column block: its scale byte (returned in *sbyte) and its two
// output words. blk is the block's shared-memory address (read again only by
// the rare fix-up paths). The code of each value is the E2M1 value nearest to
// the exact |x| / d.
template <typename T>
__device__ __forceinline__ uint2 quantize_block(const Raw16<T>& raw, uint32_t blk, bool has_gs, float inv, float fac,
                                                uint32_t* sbyte) {
  const float am = amax16<T>(raw);
  float sc = __fdiv_rn(am, 6.0f);
  if (has_gs) sc = __fmul_rn(sc, inv);
  *sbyte = f32_to_e4m3_satfinite(sc);
  const float d = __fmul_rn(e4m3_to_f32(*sbyte), fac);
  if (!(d > 0.0f)) return make_uint2(0u, 0u);
  // d below 2^-100: the comparisons need scaling (and below 2^-127 the
  // reciprocal overflows)
  if (d < 0x1p-100f) return exact_block<T>(blk, d);
  // Each value is converted twice, from x * r (1 - 2^-22) and x * r (1 +
  // 2^-22), r = 1 / d rounded: x * r is within two roundings (2^-23
  // relative) of the quotient x / d, and each bracketing product within two
  // more of x * r (1 -+ 2^-22), so the quotient lies strictly between them.
  // Where both convert to the same code (the nearest-value code is monotone)
  // that code is the one of the quotient. Codes that differ (a midpoint lies
  // between the products, or on one of them) take the exact comparisons. One
  // output word (eight values) at a time, to keep few values live.
  const float r = __frcp_rn(d);
  const float rl = __fmul_rn(r, 1.0f - 0x1p-22f), rh = __fmul_rn(r, 1.0f + 0x1p-22f);
  uint32_t hw[2], dm[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float ul[4], uh[4], vl[4], vh[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pair_at<T>(raw, 4 * h + i, ul[i], uh[i]);
      vl[i] = ul[i];
      vh[i] = uh[i];
      mul2_rn(ul[i], uh[i], rh);
      mul2_rn(vl[i], vh[i], rl);
    }
    hw[h] = cvt_e2m1x8(ul, uh);
    dm[h] = hw[h] ^ cvt_e2m1x8(vl, vh);
  }
  if (dm[0] | dm[1]) fix_codes<T>(hw[0], hw[1], dm[0], dm[1], blk, d);
  return make_uint2(plus_zero(hw[0]), plus_zero(hw[1]));
}

// The quantizer: the copy engine streams the activations into shared memory, so that the bytes in flight no longer depend on registers. Chunks
// of kQBlocks blocks of one expert's plane go through a ring of stages; one
// producer thread issues the bulk loads, eight consumer warps quantize each
// chunk (two blocks per thread) and store the words and scale bytes
// directly (a warp's stores are 256 and 32 contiguous bytes). CTA (bx, by)
// takes chunks bx, bx + gx, ... of experts by, by + gy, ...
constexpr int kQBlocks = 512;
constexpr int kQConsumers = 256;
constexpr int kQThreads = kQConsumers + 32;
template <typename T> struct QRing {
  static constexpr int kStages = sizeof(T) == 4 ? 3 : 4;
  static constexpr uint32_t kStage = kQBlocks * 16 * (uint32_t)sizeof(T);
};

template <typename T>
__global__ void __launch_bounds__(kQThreads)
quantize_kernel(const T* __restrict__ x, const float* __restrict__ gs, int64_t E, int64_t bpe,
                     uint32_t* __restrict__ w, uint8_t* __restrict__ scales) {
  using R = QRing<T>;
  extern __shared__ __align__(128) uint8_t qbuf[];
  __shared__ __align__(8) uint64_t bars[2 * R::kStages];  // full[s], then empty[s]
  __shared__ int abort_flag;
  const int warp = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
  const uint32_t sbuf = pipe::smem_addr(qbuf), sbar = pipe::smem_addr(bars);
  auto full = [&](int st) { return sbar + 8u * (uint32_t)st; };
  auto empty = [&](int st) { return sbar + 8u * (uint32_t)(R::kStages + st); };
  if (threadIdx.x == 0) {
    for (int st = 0; st < R::kStages; ++st) {
      pipe::mbar_init(full(st), 1);
      pipe::mbar_init(empty(st), kQConsumers / 32);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int64_t nch = (bpe + kQBlocks - 1) / kQBlocks;  // chunks per expert
  if (warp == kQConsumers / 32) {
    if (lane == 0) {
      int64_t it = 0;
      bool ok = true;
      for (int64_t e = blockIdx.y; e < E && ok; e += gridDim.y)
        for (int64_t c = blockIdx.x; c < nch; c += gridDim.x, ++it) {
          const int st = (int)(it % R::kStages);
          const uint32_t ph = (uint32_t)((it / R::kStages) & 1);
          // stage st is free once every consumer warp released its last use
          if (it >= R::kStages && !pipe::wait_bar(empty(st), ph ^ 1u, &abort_flag, 43, &g_copy_error)) {
            ok = false;
            break;
          }
          const int64_t b0 = c * kQBlocks;
          const uint32_t bytes = (uint32_t)((bpe - b0 < kQBlocks ? bpe - b0 : kQBlocks) * 16 * (int64_t)sizeof(T));
          pipe::mbar_arrive_tx(full(st), bytes);
          bulk_g2s(sbuf + (uint32_t)st * R::kStage, x + 16 * (e * bpe + b0), bytes, full(st));
        }
      // no copy may still be landing when the CTA exits
      for (int64_t i = it > R::kStages ? it - R::kStages : 0; i < it; ++i)
        pipe::wait_bar_quiet(full((int)(i % R::kStages)), (uint32_t)((i / R::kStages) & 1));
    }
    return;
  }
  const bool has_gs = gs != nullptr;
  int64_t it = 0;
  for (int64_t e = blockIdx.y; e < E; e += gridDim.y) {
    const float fac = global_factor(gs, e);
    const float inv = has_gs ? __fdiv_rn(kGlobalScaleDivisor, __ldg(gs + e)) : 1.0f;
    for (int64_t c = blockIdx.x; c < nch; c += gridDim.x, ++it) {
      const int st = (int)(it % R::kStages);
      const uint32_t ph = (uint32_t)((it / R::kStages) & 1);
      if (!pipe::wait_bar_warp(full(st), ph, &abort_flag, 42, &g_copy_error)) return;
      const int64_t b0 = c * kQBlocks, g0 = e * bpe + b0;
      const int nb = (int)(bpe - b0 < kQBlocks ? bpe - b0 : kQBlocks);
      const uint32_t src = sbuf + (uint32_t)st * R::kStage;
      for (int j = (int)threadIdx.x; j < nb; j += kQConsumers) {
        const uint32_t blk = src + (uint32_t)j * (16u * (uint32_t)sizeof(T));
        Raw16<T> raw;
#pragma unroll
        for (int i = 0; i < (int)(sizeof(raw.q) / sizeof(uint4)); ++i)
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(raw.q[i].x), "=r"(raw.q[i].y), "=r"(raw.q[i].z), "=r"(raw.q[i].w)
                       : "r"(blk + 16u * (uint32_t)i));
        uint32_t sbyte;
        const uint2 out = quantize_block<T>(raw, blk, has_gs, inv, fac, &sbyte);
        __stcs(reinterpret_cast<uint2*>(w) + g0 + j, out);
        scales[g0 + j] = (uint8_t)sbyte;
      }
      __syncwarp();
      if (lane == 0) pipe::mbar_arrive(empty(st));
    }
  }
}

// ---------------------------------------------------------------- folded-scale transcode
//
// The alternative that issue #693 (Technical notes) rejects, built to measure
// what it loses: weight_scale * weight_scale_2 folded into each E4M3 byte, no
// sidecar. Weight bytes are copied as they are (the word plane is the byte
// stream); each scale byte becomes the E4M3 nearest to f32(e4m3(b) * ws2),
// ties to even, saturating at 448, small products flushed to 0 or a
// subnormal.

__device__ __forceinline__ uint32_t fold_byte(uint32_t b, float ws2) {
  return f32_to_e4m3_satfinite(__fmul_rn(e4m3_to_f32(b & 0xFFu), ws2));
}

__device__ __forceinline__ uint32_t fold_word(uint32_t v, float ws2) {
  return fold_byte(v, ws2) | (fold_byte(v >> 8, ws2) << 8) | (fold_byte(v >> 16, ws2) << 16) |
         (fold_byte(v >> 24, ws2) << 24);
}

__global__ void __launch_bounds__(kStreamThreads)
transcode_folded_kernel(const uint8_t* __restrict__ mo_w, int64_t w_bytes, const uint8_t* __restrict__ mo_ws,
                        int64_t s_bytes, const float* __restrict__ ws2p, uint8_t* __restrict__ w_out,
                        uint8_t* __restrict__ s_out) {
  const float ws2 = __ldg(ws2p);
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t wv = w_bytes >> 4, sv = s_bytes >> 4;
  const uint4* wi = reinterpret_cast<const uint4*>(mo_w);
  uint4* wo = reinterpret_cast<uint4*>(w_out);
  constexpr int kU = 4;  // loads in flight per thread
  int64_t i = tid;
  for (; i + (kU - 1) * stride < wv; i += kU * stride) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) v[u] = __ldcs(wi + i + u * stride);
#pragma unroll
    for (int u = 0; u < kU; ++u) __stcs(wo + i + u * stride, v[u]);
  }
  for (; i < wv; i += stride) __stcs(wo + i, __ldcs(wi + i));
  const uint4* si = reinterpret_cast<const uint4*>(mo_ws);
  uint4* so = reinterpret_cast<uint4*>(s_out);
  for (int64_t j = tid; j < sv; j += stride) {
    const uint4 v = __ldcs(si + j);
    __stcs(so + j, make_uint4(fold_word(v.x, ws2), fold_word(v.y, ws2), fold_word(v.z, ws2), fold_word(v.w, ws2)));
  }
  for (int64_t j = (wv << 4) + tid; j < w_bytes; j += stride) w_out[j] = mo_w[j];
  for (int64_t j = (sv << 4) + tid; j < s_bytes; j += stride) s_out[j] = (uint8_t)fold_byte(mo_ws[j], ws2);
}

}  // namespace

cudaError_t launch_transcode(const uint8_t* mo_w, int64_t w_bytes, const uint8_t* mo_ws, int64_t s_bytes,
                             const float* ws2, uint32_t* w_out, uint8_t* s_out, float* gs_out,
                             cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t smem = (size_t)kCopyBufs * kCopyChunk;
  cudaError_t e = cudaFuncSetAttribute(transcode_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  transcode_bulk_kernel<<<sms, 32, smem, st>>>(mo_w, w_bytes, mo_ws, s_bytes, ws2, reinterpret_cast<uint8_t*>(w_out),
                                              s_out, gs_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void* x, int x_dtype, const float* gs, int64_t E, int64_t N, int64_t K,
                            uint32_t* w, uint8_t* scales, cudaStream_t st) {
  // x is 16-byte aligned (the API checks), so every chunk is a legal bulk copy
  const int64_t bpe = N * (K / 16);  // 16-column blocks per expert
  const int gy = (int)(E < 65535 ? E : 65535);
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // as many CTAs as are resident at once, spread over the experts, at most
  // one per chunk of an expert
  auto launch = [&](auto kern, auto* xt, uint32_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kQThreads, smem) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    const int64_t nch = (bpe + kQBlocks - 1) / kQBlocks;
    int64_t gx = ((int64_t)sms * per_sm + gy - 1) / gy;
    if (gx > nch) gx = nch;
    if (gx < 1) gx = 1;
    kern<<<dim3((unsigned)gx, (unsigned)gy), kQThreads, smem, st>>>(xt, gs, E, bpe, w, scales);
    return cudaGetLastError();
  };
  switch (x_dtype) {
    case kF32:
      return launch(quantize_kernel<float>, static_cast<const float*>(x),
                    QRing<float>::kStages * QRing<float>::kStage);
    case kF16:
      return launch(quantize_kernel<__half>, static_cast<const __half*>(x),
                    QRing<__half>::kStages * QRing<__half>::kStage);
    default:
      return launch(quantize_kernel<__nv_bfloat16>, static_cast<const __nv_bfloat16*>(x),
                    QRing<__nv_bfloat16>::kStages * QRing<__nv_bfloat16>::kStage);
  }
}

cudaError_t launch_transcode_folded(const uint8_t* mo_w, int64_t w_bytes, const uint8_t* mo_ws, int64_t s_bytes,
                                    const float* ws2, uint32_t* w_out, uint8_t* s_out, cudaStream_t st) {
  const int64_t units = (w_bytes >> 4) / 4 + (s_bytes >> 4) + 16;
  transcode_folded_kernel<<<stream_grid(transcode_folded_kernel, units), kStreamThreads, 0, st>>>(
      mo_w, w_bytes, mo_ws, s_bytes, ws2, reinterpret_cast<uint8_t*>(w_out), s_out);
  return cudaGetLastError();
}

int read_copy_error() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_copy_error, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  cudaMemcpyToSymbol(g_copy_error, &zero, sizeof(int));
  return v;
}

cudaError_t launch_dequantize(const uint32_t* w, const uint8_t* scales, const float* gs, int64_t E,
                              int64_t N, int64_t K, int out_dtype, void* out, cudaStream_t st) {
  const int64_t gpe = N * (K / 8);  // words per expert
  auto grid_of = [&](auto kern) {
    int gx = stream_grid(kern, (gpe * E + 7) / 8);
    const int64_t per_expert = (gpe + kStreamThreads - 1) / kStreamThreads;
    if (gx > per_expert) gx = (int)(per_expert < 1 ? 1 : per_expert);
    const int gy = (int)(E < 65535 ? E : 65535);
    return dim3(gx, gy);
  };
  switch (out_dtype) {
    case kF32:
      dequantize_kernel<float><<<grid_of(dequantize_kernel<float>), kStreamThreads, 0, st>>>(w, scales, gs, E, gpe,
                                                                                            (float*)out);
      break;
    case kF16:
      dequantize_kernel<__half><<<grid_of(dequantize_kernel<__half>), kStreamThreads, 0, st>>>(w, scales, gs, E, gpe,
                                                                                              (__half*)out);
      break;
    default:
      dequantize_kernel<__nv_bfloat16><<<grid_of(dequantize_kernel<__nv_bfloat16>), kStreamThreads, 0, st>>>(
          w, scales, gs, E, gpe, (__nv_bfloat16*)out);
      break;
  }
  return cudaGetLastError();
}

}  // namespace nvfp4
