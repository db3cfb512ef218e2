// Decode-size QuantizedMatmul with a non-transposed weight (mlx PR #2629,
// Changes during review: the quantized axis of such a weight is N): y = x @
// dequantize(w) * gs / 2688 for up to sixteen token rows, w [K, N/8] words
// (word j of row k holds outputs 8j..8j+7 of input k, nibble i output 8j+i),
// one E4M3 byte per 16 outputs of an input.
//
// The weight plane is streamed once per eight token rows, through m16n8k16
// MMAs: A is the weight (rows = outputs, columns = inputs), B the activations
// (eight token columns). An MMA wants each register's two f16 values to be
// neighbours along K, while a word holds neighbours along N; so the words of
// two input rows are interleaved nibble by nibble (two shifts and two logic
// ops give two words whose bytes are (row k, row k+1) code pairs), and one
// E2M1x2 conversion then yields the pair the MMA expects. The scale pair of
// those two rows multiplies it (fp4 * e4m3 is exact in f16). A lane (g, t)
// owns inputs 4t..4t+3 of every 16-input step and word columns 4g..4g+3 of
// its warp's 32-word slab; MMA p of column c puts output 8j+2p in row g and
// 8j+2p+1 in row g+8. Every lane thus decodes each word it loads exactly
// once, with no data exchanged between lanes.
//
// Work is a flat list of 16-input steps, slab by slab; each warp takes one
// contiguous run of it (the runs differ by at most one step) and streams it
// through its own ring of shared-memory stages filled by per-lane cp.async
// copies (weights 2 KB, scale bytes 256 B and activations 256 B a step;
// planes whose rows or bases do not meet the copy alignment are loaded and
// stored instead). A run that leaves a slab, or ends, adds its sums into a
// float workspace [M, N] (red.global.add.v4.f32); a second kernel scales,
// rounds and writes y, and returns the workspace to zero for the next call.
//
// bf16 activations take the f16 MMA when a step's values convert to f16
// exactly (checked per step, warp-wide); otherwise that step decodes the
// weights to bf16 and runs the bf16 MMA on the raw activations.
#include <cstdint>
#include <map>
#include <mutex>
#include <type_traits>
#include <vector>

#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_qmv_common.cuh"

namespace nvfp4 {

namespace {

constexpr int kNtThreads = 256;  // eight warps, each with its own ring
constexpr int kNtWarps = kNtThreads / 32;
constexpr int kNtStages = 4;       // 16-input steps in flight per warp
constexpr int kNtSlabWords = 32;   // word columns per warp slab (256 outputs)
constexpr int kNtMinSteps = 3;     // fewest steps a warp is given (when the plane is small)
// One stage: weight words in 16-byte units (rows 4t+r, columns 4g..4g+3) at
// unit nt_word_unit(r, t, g), scale bytes [16 rows][16 groups] (row 4t+r at
// position 4r+t, so a lane's four rows fall in distinct banks), activations
// [lane] (8 B: token g, inputs 4t..4t+3).
constexpr uint32_t kNtWordBytes = 2048, kNtScaleBytes = 256, kNtXBytes = 256;
constexpr uint32_t kNtStageBytes = kNtWordBytes + kNtScaleBytes + kNtXBytes;
constexpr uint32_t kNtSmem = kNtWarps * kNtStages * kNtStageBytes;

// Unit (r*4 + t)*8 + (g ^ 2t): the eight lanes that copy one 128-byte row
// segment (same t, g = 0..7) write eight distinct bank groups, and so do the
// eight lanes of each quarter-warp phase of the 16-byte fragment reads
// (g in {2q, 2q+1}, t = 0..3).
__device__ __forceinline__ uint32_t nt_word_unit(int r, int t, int g) {
  return (uint32_t)((r * 4 + t) * 8 + (g ^ (2 * t)));
}

struct NtArgs {
  const void* x;
  int M;
  int64_t K;
  const uint32_t* w;
  const uint8_t* scales;
  int64_t N;
  float* ws;
  int64_t ksteps;  // 16-input steps per slab
  int64_t steps;   // slabs * ksteps
  int64_t nwarps;  // warps in the grid
};

// L1-allocating copies: the eight lanes' 16-byte pieces of one 128-byte row
// segment then reach L2 as whole sectors (with .cg each half sector went to
// L2 as a request of its own, doubling the L2 reads).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// A lane's copy sources for one 16-input step of a slab: word row kb + 4t at
// column 4g of the slab, scale row kb + lane/2 at group 8 (lane & 1), and
// activation row g at input kb + 4t. Advanced by one step with three pointer
// increments; rebuilt when the run moves to the next slab. Positions are
// 32-bit on the copy path (taken only for K and N below 2^31).
template <bool kAligned>
struct NtCursor {
  using Idx = typename std::conditional<kAligned, int, int64_t>::type;
  const uint32_t* w;
  const uint8_t* s;
  const unsigned short* x;
  Idx slab, kb;
  bool col_ok, grp_ok;
};

template <bool kAligned>
__device__ __forceinline__ void nt_seek(const NtArgs& a, int64_t slab, int64_t kb, int lane, NtCursor<kAligned>& c) {
  using Idx = typename NtCursor<kAligned>::Idx;
  const int g = lane >> 2, t = lane & 3;
  const int64_t nwords = a.N / 8, ngroups = a.N / 16;
  const int64_t j = slab * kNtSlabWords + 4 * g, grp = slab * 16 + 8 * (lane & 1);
  c.slab = (Idx)slab;
  c.kb = (Idx)kb;
  c.col_ok = j < nwords;
  c.grp_ok = grp < ngroups;
  c.w = a.w + (kb + 4 * t) * nwords + j;
  c.s = a.scales + (kb + (lane >> 1)) * ngroups + grp;
  c.x = static_cast<const unsigned short*>(a.x) + (int64_t)g * a.K + kb + 4 * t;
}

template <bool kAligned>
__device__ __forceinline__ void nt_advance(const NtArgs& a, int lane, NtCursor<kAligned>& c) {
  c.kb += 16;
  if (c.kb == (typename NtCursor<kAligned>::Idx)a.ksteps * 16) {
    nt_seek(a, c.slab + 1, 0, lane, c);
  } else {
    c.w += 16 * (a.N / 8);
    c.s += 16 * (a.N / 16);
    c.x += 16;
  }
}

// Copies one step's weights, scale bytes and activations into a stage
// (planes with N % 128 == 0, K % 4 == 0 and aligned bases: whole 16-byte
// word units, 8-byte scale units and 8-byte activation units, each either
// entirely inside the plane or entirely outside, where it reads as zeros).
__device__ __forceinline__ void nt_fill_copy(const NtArgs& a, const NtCursor<true>& c, uint32_t stage, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int64_t nwords = a.N / 8;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const bool ok = c.col_ok && c.kb + 4 * t + r < a.K;
    cp_async16(stage + nt_word_unit(r, t, g) * 16u, ok ? (const void*)(c.w + r * nwords) : (const void*)a.w,
               ok ? 16u : 0u);
  }
  {
    const int rho = lane >> 1;
    const bool ok = c.grp_ok && c.kb + rho < a.K;
    cp_async8(stage + kNtWordBytes + (uint32_t)((4 * (rho & 3) + (rho >> 2)) * 16 + 8 * (lane & 1)),
              ok ? (const void*)c.s : (const void*)a.scales, ok ? 8u : 0u);
  }
  {
    const bool ok = g < a.M && c.kb + 4 * t < a.K;
    cp_async8(stage + kNtWordBytes + kNtScaleBytes + (uint32_t)lane * 8u, ok ? (const void*)c.x : a.x, ok ? 8u : 0u);
  }
}

// The same stage contents from plain loads, for any plane: rows past K,
// columns past N/8 and token rows past M are zeros.
__device__ __forceinline__ void nt_fill_plain(const NtArgs& a, const NtCursor<false>& c, uint32_t stage, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int64_t nwords = a.N / 8, ngroups = a.N / 16, kb = c.kb;
  const int64_t j = c.slab * kNtSlabWords + 4 * g;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t k = kb + 4 * t + r;
    uint32_t v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = k < a.K && j + q < nwords ? __ldg(a.w + k * nwords + j + q) : 0u;
    sts128(stage + nt_word_unit(r, t, g) * 16u, v[0], v[1], v[2], v[3]);
  }
  {  // scale bytes: row kb + rho, groups 16 slab + 8h .. + 7
    const int rho = lane >> 1, h = lane & 1;
    const int64_t k = kb + rho, grp = c.slab * 16 + 8 * h;
    uint32_t v[2] = {0u, 0u};
#pragma unroll
    for (int b = 0; b < 8; ++b)
      if (k < a.K && grp + b < ngroups) v[b >> 2] |= (uint32_t)__ldg(a.scales + k * ngroups + grp + b) << (8 * (b & 3));
    sts64(stage + kNtWordBytes + (uint32_t)((4 * (rho & 3) + (rho >> 2)) * 16 + 8 * h), v[0], v[1]);
  }
  {  // activations: token g, inputs kb + 4t .. + 3
    const int64_t k = kb + 4 * t;
    const unsigned short* xs = static_cast<const unsigned short*>(a.x);
    uint32_t v[2] = {0u, 0u};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (g < a.M && k + q < a.K) v[q >> 1] |= (uint32_t)__ldg(xs + g * a.K + k + q) << (16 * (q & 1));
    sts64(stage + kNtWordBytes + kNtScaleBytes + (uint32_t)lane * 8u, v[0], v[1]);
  }
}

template <bool kAligned>
__device__ __forceinline__ void nt_fill(const NtArgs& a, const NtCursor<kAligned>& c, uint32_t stage, int lane) {
  if constexpr (kAligned)
    nt_fill_copy(a, c, stage, lane);
  else
    nt_fill_plain(a, c, stage, lane);
}

// Two E4M3 bytes -> bf16x2 of scale * 2^112 (exact: four significant bits;
// the bf16 decode of the codes carries the matching 2^-112).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_x2p112(uint32_t two_bytes) {
  const uint32_t h = e4m3x2_to_f16x2(two_bytes);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * 0x1p112f, f.y * 0x1p112f);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Sixteen MMAs of one step in operand type U (f16, or bf16 when the step's
// activations do not fit f16). wr[r] = the lane's four words of input row
// 4t+r; sc[r] = its two scale bytes of that row (groups of columns 0-1 and
// 2-3).
template <typename U>
__device__ __forceinline__ void nt_mma(const uint4 (&wr)[4], const uint32_t (&sc)[4], uint32_t b0, uint32_t b1,
                                       float (&acc)[4][4][4]) {
  uint32_t s01[2], s23[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t sel = h ? 0x0051u : 0x0040u;  // (row a byte h, row b byte h)
    const uint32_t p01 = __byte_perm(sc[0], sc[1], sel), p23 = __byte_perm(sc[2], sc[3], sel);
    if constexpr (std::is_same<U, __half>::value) {
      s01[h] = e4m3x2_to_f16x2(p01);
      s23[h] = e4m3x2_to_f16x2(p23);
    } else {
      s01[h] = e4m3x2_to_bf16x2_x2p112(p01);
      s23[h] = e4m3x2_to_bf16x2_x2p112(p23);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w0 = qmv::u4get(wr[0], c), w1 = qmv::u4get(wr[1], c);
    const uint32_t w2 = qmv::u4get(wr[2], c), w3 = qmv::u4get(wr[3], c);
    // byte p of e: (nibble 2p of the first row, nibble 2p of the second);
    // of o: the same for nibble 2p+1
    const uint32_t e01 = (w0 & 0x0F0F0F0Fu) | ((w1 << 4) & 0xF0F0F0F0u);
    const uint32_t o01 = ((w0 >> 4) & 0x0F0F0F0Fu) | (w1 & 0xF0F0F0F0u);
    const uint32_t e23 = (w2 & 0x0F0F0F0Fu) | ((w3 << 4) & 0xF0F0F0F0u);
    const uint32_t o23 = ((w2 >> 4) & 0x0F0F0F0Fu) | (w3 & 0xF0F0F0F0u);
    uint32_t de01[4], do01[4], de23[4], do23[4];
    Dt<U>::decode(e01, s01[c >> 1], de01);
    Dt<U>::decode(o01, s01[c >> 1], do01);
    Dt<U>::decode(e23, s23[c >> 1], de23);
    Dt<U>::decode(o23, s23[c >> 1], do23);
#pragma unroll
    for (int p = 0; p < 4; ++p) qmv::MmaOp<U>::run(acc[c][p], de01[p], do01[p], de23[p], do23[p], b0, b1);
  }
}

template <typename T>
__device__ __forceinline__ void nt_step(uint32_t stage, int lane, float (&acc)[4][4][4]) {
  const int g = lane >> 2, t = lane & 3;
  uint4 wr[4];
  uint32_t sc[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    wr[r] = qmv::lds128(stage + nt_word_unit(r, t, g) * 16u);
    sc[r] = lds_u16(stage + kNtWordBytes + (uint32_t)((4 * r + t) * 16 + 2 * g));
  }
  const uint2 xv = lds64(stage + kNtWordBytes + kNtScaleBytes + (uint32_t)lane * 8u);
  if constexpr (std::is_same<T, __half>::value) {
    nt_mma<__half>(wr, sc, xv.x, xv.y, acc);
  } else {
    const uint32_t in[2] = {xv.x, xv.y};
    uint32_t o[2];
    int inexact = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const float lo = __uint_as_float(in[p] << 16), hi = __uint_as_float(in[p] & 0xFFFF0000u);
      const __half2 h = __floats2half2_rn(lo, hi);
      const float2 back = __half22float2(h);
      inexact |= (back.x != lo) | (back.y != hi);
      o[p] = *reinterpret_cast<const uint32_t*>(&h);
    }
    if (__any_sync(0xffffffffu, inexact))
      nt_mma<__nv_bfloat16>(wr, sc, xv.x, xv.y, acc);
    else
      nt_mma<__half>(wr, sc, o[0], o[1], acc);
  }
}

// Adds the run's sums for one slab into the workspace and clears them. Lane
// (g, t) holds tokens 2t and 2t+1 of word columns 4g..4g+3: output 8j+2p in
// acc[c][p][token & 1], 8j+2p+1 in acc[c][p][2 + (token & 1)].
__device__ __forceinline__ void nt_flush(const NtArgs& a, int64_t slab, int lane, float (&acc)[4][4][4]) {
  const int g = lane >> 2, t = lane & 3;
  const int64_t nwords = a.N / 8;
#pragma unroll
  for (int tk = 0; tk < 2; ++tk) {
    const int m = 2 * t + tk;
    if (m < a.M) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t j = slab * kNtSlabWords + 4 * g + c;
        if (j < nwords) {
          float* dst = a.ws + (int64_t)m * a.N + 8 * j;
          red_add_v4(dst, acc[c][0][tk], acc[c][0][2 + tk], acc[c][1][tk], acc[c][1][2 + tk]);
          red_add_v4(dst + 4, acc[c][2][tk], acc[c][2][2 + tk], acc[c][3][tk], acc[c][3][2 + tk]);
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][p][i] = 0.0f;
}

// One warp's run of steps s0..s1-1 through its ring: acc collects a slab's
// sums, which go to the workspace when the slab or the run ends.
template <typename T, bool kAligned>
__device__ __forceinline__ void nt_run(const NtArgs& a, int64_t s0, int64_t s1, uint32_t ring, int lane) {
  int64_t slab = s0 / a.ksteps;
  const int64_t slab_end = (slab + 1) * a.ksteps;
  NtCursor<kAligned> cur;  // the next step to fill
  nt_seek(a, slab, (s0 - slab * a.ksteps) * 16, lane, cur);
#pragma unroll
  for (int i = 0; i < kNtStages; ++i) {
    if (s0 + i < s1) {
      nt_fill<kAligned>(a, cur, ring + (uint32_t)i * kNtStageBytes, lane);
      nt_advance(a, lane, cur);
    }
    cp_commit();  // one group per step, empty ones included, so the wait count is fixed
  }
  // left: steps of the run still to compute (this one included); to_end:
  // steps until the current slab ends, capped by left (a run is far below
  // 2^31 steps)
  int left = (int)(s1 - s0), to_end = (int)(slab_end - s0 < s1 - s0 ? slab_end - s0 : s1 - s0);
  float acc[4][4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][p][i] = 0.0f;
  int slot = 0;
  for (; left > 0; --left) {
    const uint32_t stage = ring + (uint32_t)slot * kNtStageBytes;
    cp_wait<kNtStages - 1>();  // this step's group has landed
    __syncwarp();              // and so have the other lanes' (the scale bytes are shared)
    nt_step<T>(stage, lane, acc);
    if (--to_end == 0) {  // the slab or the run ends here
      nt_flush(a, slab, lane, acc);
      ++slab;
      to_end = (int)(a.ksteps < left - 1 ? a.ksteps : left - 1);
    }
    __syncwarp();  // every lane is done with the stage before it is refilled
    if (left > kNtStages) {
      nt_fill<kAligned>(a, cur, stage, lane);
      nt_advance(a, lane, cur);
    }
    cp_commit();
    slot = slot + 1 == kNtStages ? 0 : slot + 1;
  }
  cp_wait<0>();
}

// Work is a flat list of 16-input steps, slab by slab; warp gw of the grid
// takes one contiguous run of it (the runs differ by at most one step).
template <typename T, bool kAligned>
__global__ void __launch_bounds__(kNtThreads, 2) qmv_nt_kernel(const NtArgs a) {
  extern __shared__ __align__(16) uint8_t nt_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * kNtWarps + warp;
  const int64_t q = a.steps / a.nwarps, rem = a.steps % a.nwarps;
  const int64_t s0 = gw * q + (gw < rem ? gw : rem), s1 = s0 + q + (gw < rem ? 1 : 0);
  if (s0 >= s1) return;  // warp-uniform
  nt_run<T, kAligned>(a, s0, s1,
                      (uint32_t)__cvta_generic_to_shared(nt_smem) + (uint32_t)warp * kNtStages * kNtStageBytes, lane);
}

// y = cast(ws * gs / 2688); the workspace returns to zero.
template <typename T>
__global__ void __launch_bounds__(256) qmv_nt_finish(float* __restrict__ ws, int64_t n, const float* __restrict__ gs,
                                                     T* __restrict__ y) {
  const float fac = global_factor(gs, 0);
  const bool has_gs = gs != nullptr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = ws[i];
    ws[i] = 0.0f;
    y[i] = from_f32<T>(has_gs ? __fmul_rn(v, fac) : v);
  }
}

// Float workspace [kQmvNtMaxM, N] per (device, stream), zero when handed
// out; grown on demand (a new buffer is zeroed on the calling stream, so a
// captured call zeroes it in every replay) and kept until
// release_nt_workspaces().
std::mutex g_nt_mu;
std::map<std::pair<int, uintptr_t>, std::pair<float*, size_t>> g_nt;
std::vector<float*> g_nt_retired;

cudaError_t nt_workspace(int dev, cudaStream_t st, size_t floats, float** out) {
  std::lock_guard<std::mutex> lock(g_nt_mu);
  auto& slot = g_nt[{dev, reinterpret_cast<uintptr_t>(st)}];
  if (slot.second < floats) {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaError_t e = cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) return e;
    float* ptr = nullptr;
    e = cudaMalloc(&ptr, floats * sizeof(float));
    cudaStreamCaptureMode back = mode;
    cudaThreadExchangeStreamCaptureMode(&back);
    if (e != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(ptr, 0, floats * sizeof(float), st)) != cudaSuccess) return e;
    if (slot.first) g_nt_retired.push_back(slot.first);
    slot = {ptr, floats};
  }
  *out = slot.first;
  return cudaSuccess;
}

template <typename T, bool kAligned>
cudaError_t launch_kernel(NtArgs a, int sms, cudaStream_t st) {
  auto kern = qmv_nt_kernel<T, kAligned>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kNtSmem);
  if (e != cudaSuccess) return e;
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kNtThreads, kNtSmem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t want = (a.steps + kNtWarps * kNtMinSteps - 1) / (kNtWarps * kNtMinSteps), cap = (int64_t)sms * per_sm;
  const int64_t ctas = want < cap ? want : cap;
  a.nwarps = ctas * kNtWarps;
  kern<<<(unsigned)ctas, kNtThreads, kNtSmem, st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const void* x, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales, const float* gs,
                     int64_t N, void* y, cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  float* ws = nullptr;
  cudaError_t e = nt_workspace(dev, st, (size_t)kQmvNtMaxM * (size_t)N, &ws);
  if (e != cudaSuccess) return e;
  // copies need 16-byte word rows in whole 4-word units, 8-byte scale rows in
  // whole 8-byte units and 8-byte activation units
  const bool aligned = N % 128 == 0 && K % 4 == 0 && N < (1ll << 31) && K < (1ll << 30) &&
                       reinterpret_cast<uintptr_t>(w) % 16 == 0 && reinterpret_cast<uintptr_t>(scales) % 8 == 0 &&
                       reinterpret_cast<uintptr_t>(x) % 8 == 0;
  // one pass per eight token rows (the MMA's eight B columns); a second pass
  // reads the plane again
  for (int64_t m0 = 0; m0 < M; m0 += 8) {
    const int64_t mp = M - m0 < 8 ? M - m0 : 8;
    NtArgs a{static_cast<const T*>(x) + m0 * K, (int)mp, K, w, scales, N, ws + m0 * N, (K + 15) / 16, 0, 0};
    a.steps = (N / 8 + kNtSlabWords - 1) / kNtSlabWords * a.ksteps;
    e = aligned ? launch_kernel<T, true>(a, sms, st) : launch_kernel<T, false>(a, sms, st);
    if (e != cudaSuccess) return e;
  }
  const int64_t n = M * N, fb = (n + 255) / 256;
  qmv_nt_finish<T><<<(unsigned)(fb < 4 * sms ? fb : 4 * sms), 256, 0, st>>>(ws, n, gs, static_cast<T*>(y));
  return cudaGetLastError();
}

}  // namespace

bool qmv_nt_supported(int64_t M, int64_t N, int64_t K) {
  return M >= 1 && M <= kQmvNtMaxM && N > 0 && N % 16 == 0 && K > 0 && N < (1ll << 40) && K < (1ll << 40);
}

cudaError_t launch_qmv_nt(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                          const float* gs, int64_t N, void* y, cudaStream_t st) {
  if (xdt == kBF16) return launch_t<__nv_bfloat16>(x, M, K, w, scales, gs, N, y, st);
  return launch_t<__half>(x, M, K, w, scales, gs, N, y, st);
}

void release_nt_workspaces() {
  std::lock_guard<std::mutex> lock(g_nt_mu);
  for (auto& kv : g_nt) cudaFree(kv.second.first);
  g_nt.clear();
  for (float* p : g_nt_retired) cudaFree(p);
  g_nt_retired.clear();
}

}  // namespace nvfp4
