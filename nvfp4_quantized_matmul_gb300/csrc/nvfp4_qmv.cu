// Decode-shape NVFP4 products: y[r, n] = factor(e_r) * sum_k x[lhs_r, k] * deq(w[e_r])[n, k].
//
// QuantizedMatmul below the tensor-core crossover and every GatherQMM decode
// (mlxcel PR #2629 "ROCm native NVFP4", Summary: one pass per output block,
// global scale applied once per output; Changes during review: out-of-range
// expert rows are exact zeros).
//
// GB300 design. The work is bound by streaming the packed weights (9/16 byte
// per element), but at HBM rate the SIMT pipes leave only ~3 instructions per
// weight element, too few to decode and FMA in f32 for more than one token.
// So the weight fragment is decoded straight into registers in the
// m16n8k16 A-operand layout and the tokens ride in the 8-wide B operand; the
// tensor pipe does the multiply-accumulate in f32 and the decode is paid once
// per weight element regardless of the token count.
//
// Tiling: a CTA owns 16 weight rows and up to 8*MT output rows; its eight
// warps split K (128-column chunks) and reduce through shared memory, so no
// global scratch is needed. Lane (g = lane/4, t = lane%4) streams words
// 4t..4t+3 of rows g and g+8 of each chunk with one 128-bit load per row.
// K positions inside one MMA are a permutation of the chunk's columns: in
// k16-step s lane t's A slots {2t, 2t+1, 2t+8, 2t+9} hold columns 32t+4s+0..3,
// and its B slots take the activations of those same columns, so each lane's
// activations for a chunk are 32 contiguous elements.
#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <typename XT> struct MmaOp;
template <> struct MmaOp<__half> {
  __device__ static __forceinline__ void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
};
template <> struct MmaOp<__nv_bfloat16> {
  __device__ static __forceinline__ void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
};

template <int MT>
struct Chunk {
  uint4 wa, wb;     // words 4t..4t+3 of rows g and g+8
  uint32_t sa, sb;  // scale bytes of groups 2t, 2t+1 (low 16 bits) of rows g and g+8
  uint4 xv[MT][4];  // activations of token slot g+8*mt, columns 32t..32t+31 of the chunk
};

struct Pass {
  const uint32_t* row_g;   // packed row n0+g of the expert (null if n >= N)
  const uint32_t* row_g8;  // packed row n0+g+8
  const uint8_t* sc_g;
  const uint8_t* sc_g8;
  int64_t kwords, kgroups, K;
};

template <typename XT, int MT, bool VEC>
__device__ __forceinline__ void load_chunk(Chunk<MT>& ch, int64_t c, const Pass& p, const XT* const (&xrow)[MT],
                                           int t) {
  const int64_t kw = c * 16 + 4 * t;
  const int64_t gi = c * 8 + 2 * t;
  if (VEC) {  // K % 32 == 0: a lane's four words (and two scales) are all in range or all out
    const bool ok = kw < p.kwords;
    ch.wa = (ok && p.row_g) ? ld_stream_v4(p.row_g + kw) : make_uint4(0, 0, 0, 0);
    ch.wb = (ok && p.row_g8) ? ld_stream_v4(p.row_g8 + kw) : make_uint4(0, 0, 0, 0);
    ch.sa = (ok && p.row_g) ? (uint32_t)__ldcs(reinterpret_cast<const unsigned short*>(p.sc_g + gi)) : 0u;
    ch.sb = (ok && p.row_g8) ? (uint32_t)__ldcs(reinterpret_cast<const unsigned short*>(p.sc_g8 + gi)) : 0u;
  } else {  // K % 32 == 16: words come in in-range pairs (one 16-column block each)
    const bool ok0 = kw < p.kwords, ok1 = kw + 2 < p.kwords;
    uint2 a0 = make_uint2(0, 0), a1 = a0, b0 = a0, b1 = a0;
    uint32_t sa = 0, sb = 0;
    if (p.row_g) {
      if (ok0) { a0 = ld_stream_v2(p.row_g + kw); sa = p.sc_g[gi]; }
      if (ok1) { a1 = ld_stream_v2(p.row_g + kw + 2); sa |= (uint32_t)p.sc_g[gi + 1] << 8; }
    }
    if (p.row_g8) {
      if (ok0) { b0 = ld_stream_v2(p.row_g8 + kw); sb = p.sc_g8[gi]; }
      if (ok1) { b1 = ld_stream_v2(p.row_g8 + kw + 2); sb |= (uint32_t)p.sc_g8[gi + 1] << 8; }
    }
    ch.wa = make_uint4(a0.x, a0.y, a1.x, a1.y);
    ch.wb = make_uint4(b0.x, b0.y, b1.x, b1.y);
    ch.sa = sa;
    ch.sb = sb;
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t col = c * 128 + 32 * t + 8 * q;  // 8 columns; K % 16 == 0 keeps them all in or out
      ch.xv[mt][q] = (xrow[mt] && col < p.K) ? __ldg(reinterpret_cast<const uint4*>(xrow[mt] + col))
                                             : make_uint4(0, 0, 0, 0);
    }
  }
}

__device__ __forceinline__ uint32_t u4get(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <typename XT, int MT>
__device__ __forceinline__ void compute_chunk(const Chunk<MT>& ch, float (&acc)[MT][4]) {
  const uint32_t sa0 = Dt<XT>::scale(ch.sa & 0xFF), sa1 = Dt<XT>::scale((ch.sa >> 8) & 0xFF);
  const uint32_t sb0 = Dt<XT>::scale(ch.sb & 0xFF), sb1 = Dt<XT>::scale((ch.sb >> 8) & 0xFF);
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // word j of the lane: columns 32t+8j..+7, k16-steps 2j and 2j+1
    uint32_t da[4], db[4];
    Dt<XT>::decode(u4get(ch.wa, j), j < 2 ? sa0 : sa1, da);
    Dt<XT>::decode(u4get(ch.wb, j), j < 2 ? sb0 : sb1, db);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int s = 2 * j + h;  // bytes 2h, 2h+1 of the word feed step s
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint32_t b0 = u4get(ch.xv[mt][(2 * s) >> 2], (2 * s) & 3);
        const uint32_t b1 = u4get(ch.xv[mt][(2 * s + 1) >> 2], (2 * s + 1) & 3);
        MmaOp<XT>::run(acc[mt], da[2 * h], db[2 * h], da[2 * h + 1], db[2 * h + 1], b0, b1);
      }
    }
  }
}

template <typename XT, int MT, bool VEC>
__global__ void __launch_bounds__(kThreads)
qmv_mma_kernel(const QmvArgs a) {
  constexpr int TR = 8 * MT;  // output rows (token slots) per CTA
  __shared__ int64_t s_e[TR];
  __shared__ int64_t s_x[TR];
  __shared__ float s_red[kWarps][MT][4][32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t n0 = (int64_t)blockIdx.x * 16;
  const int64_t r0 = (int64_t)blockIdx.y * TR;
  const XT* x = static_cast<const XT*>(a.x);

  if (threadIdx.x < TR) {
    const int64_t r = r0 + threadIdx.x;
    int64_t e = -1, xr = -1;
    if (r < a.R) {
      e = a.rhs ? (int64_t)a.rhs[r] : 0;
      xr = a.lhs ? (int64_t)a.lhs[r] : r;
      if (e >= a.E || xr >= a.B) e = -1;  // zero row
    }
    s_e[threadIdx.x] = e;
    s_x[threadIdx.x] = xr;
  }
  __syncthreads();

  const int64_t nchunks = (a.K + 127) / 128;
  const int64_t c_begin = nchunks * warp / kWarps, c_end = nchunks * (warp + 1) / kWarps;

  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;

  uint32_t pending = 0;
  for (int j = 0; j < TR; ++j)
    if (s_e[j] >= 0) pending |= 1u << j;

  const int64_t kwords = a.K / 8, kgroups = a.K / 16;
  while (pending) {  // one pass per distinct expert among the CTA's rows
    const int first = __ffs(pending) - 1;
    const int64_t e = s_e[first];
    uint32_t mask = 0;
    for (int j = 0; j < TR; ++j)
      if (((pending >> j) & 1) && s_e[j] == e) mask |= 1u << j;
    pending &= ~mask;

    Pass p;
    const int64_t ng = n0 + g, ng8 = n0 + g + 8;
    const uint32_t* wexp = a.w + e * a.N * kwords;
    const uint8_t* sexp = a.scales + e * a.N * kgroups;
    p.row_g = ng < a.N ? wexp + ng * kwords : nullptr;
    p.row_g8 = ng8 < a.N ? wexp + ng8 * kwords : nullptr;
    p.sc_g = sexp + ng * kgroups;
    p.sc_g8 = sexp + ng8 * kgroups;
    p.kwords = kwords;
    p.kgroups = kgroups;
    p.K = a.K;
    const XT* xrow[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int slot = g + 8 * mt;
      xrow[mt] = ((mask >> slot) & 1) ? x + s_x[slot] * a.K : nullptr;
    }

    // Three register stages: two chunks in flight while one is decoded.
    Chunk<MT> c0, c1, c2;
    int64_t c = c_begin;
    if (c < c_end) load_chunk<XT, MT, VEC>(c0, c, p, xrow, t);
    if (c + 1 < c_end) load_chunk<XT, MT, VEC>(c1, c + 1, p, xrow, t);
    for (; c < c_end; c += 3) {
      if (c + 2 < c_end) load_chunk<XT, MT, VEC>(c2, c + 2, p, xrow, t);
      compute_chunk<XT, MT>(c0, acc);
      if (c + 1 >= c_end) break;
      if (c + 3 < c_end) load_chunk<XT, MT, VEC>(c0, c + 3, p, xrow, t);
      compute_chunk<XT, MT>(c1, acc);
      if (c + 2 >= c_end) break;
      if (c + 4 < c_end) load_chunk<XT, MT, VEC>(c1, c + 4, p, xrow, t);
      compute_chunk<XT, MT>(c2, acc);
    }
  }

  // Reduce the eight K-slices.
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) s_red[warp][mt][i][lane] = acc[mt][i];
  __syncthreads();
  XT* y = static_cast<XT*>(a.y);
  for (int idx = threadIdx.x; idx < MT * 4 * 32; idx += kThreads) {
    const int l = idx & 31, i = (idx >> 5) & 3, mt = idx >> 7;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += s_red[w][mt][i][l];
    // D fragment: c0,c1 -> (row g, tokens 2t, 2t+1); c2,c3 -> (row g+8, same tokens)
    const int lg = l >> 2, lt = l & 3;
    const int64_t n = n0 + lg + ((i & 2) ? 8 : 0);
    const int slot = 8 * mt + 2 * lt + (i & 1);
    const int64_t r = r0 + slot;
    if (n >= a.N || r >= a.R) continue;
    const int64_t e = s_e[slot];
    const float out = e < 0 ? 0.f : (a.gs ? __fmul_rn(v, global_factor(a.gs, e)) : v);
    y[r * a.N + n] = Dt<XT>::from_f32(out);
  }
}

// f32 activations: exact-product SIMT path (one warp per weight row and up
// to four output rows; lanes stride over the packed words, shuffle reduce).
constexpr int kF32Tokens = 4;
__global__ void __launch_bounds__(kThreads)
qmv_f32_kernel(const QmvArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t r0 = (int64_t)blockIdx.y * kF32Tokens;
  if (n >= a.N) return;
  const float* x = static_cast<const float*>(a.x);
  int64_t e[kF32Tokens], xr[kF32Tokens];
#pragma unroll
  for (int j = 0; j < kF32Tokens; ++j) {
    const int64_t r = r0 + j;
    e[j] = -1;
    xr[j] = 0;
    if (r < a.R) {
      const int64_t ee = a.rhs ? (int64_t)a.rhs[r] : 0;
      const int64_t xx = a.lhs ? (int64_t)a.lhs[r] : r;
      if (ee < a.E && xx < a.B) { e[j] = ee; xr[j] = xx; }
    }
  }
  const int64_t kwords = a.K / 8, kgroups = a.K / 16;
  float acc[kF32Tokens];
#pragma unroll
  for (int j = 0; j < kF32Tokens; ++j) {
    acc[j] = 0.f;
    if (e[j] < 0) continue;
    const uint32_t* wr = a.w + (e[j] * a.N + n) * kwords;
    const uint8_t* sr = a.scales + (e[j] * a.N + n) * kgroups;
    const float* xp = x + xr[j] * a.K;
    for (int64_t kw = lane; kw < kwords; kw += 32) {
      uint32_t h[4];
      decode8_scaled_f16(wr[kw], e4m3_to_f16x2_bcast(sr[kw >> 1]), h);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float lo = __half2float(__ushort_as_half((unsigned short)(h[b] & 0xFFFF)));
        const float hi = __half2float(__ushort_as_half((unsigned short)(h[b] >> 16)));
        acc[j] = fmaf(xp[8 * kw + 2 * b], lo, acc[j]);
        acc[j] = fmaf(xp[8 * kw + 2 * b + 1], hi, acc[j]);
      }
    }
  }
  float* y = static_cast<float*>(a.y);
#pragma unroll
  for (int j = 0; j < kF32Tokens; ++j) {
    float v = acc[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int64_t r = r0 + j;
    if (lane == 0 && r < a.R) {
      y[r * a.N + n] = e[j] < 0 ? 0.f : (a.gs ? __fmul_rn(v, global_factor(a.gs, e[j])) : v);
    }
  }
}

template <typename XT, int MT>
cudaError_t launch_mma(const QmvArgs& a, cudaStream_t st) {
  const dim3 grid((unsigned)((a.N + 15) / 16), (unsigned)((a.R + 8 * MT - 1) / (8 * MT)));
  if (a.K % 32 == 0)
    qmv_mma_kernel<XT, MT, true><<<grid, kThreads, 0, st>>>(a);
  else
    qmv_mma_kernel<XT, MT, false><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qmv(const QmvArgs& a, int xdt, cudaStream_t st) {
  if (xdt == kF32) {
    const dim3 grid((unsigned)((a.N + kWarps - 1) / kWarps), (unsigned)((a.R + kF32Tokens - 1) / kF32Tokens));
    qmv_f32_kernel<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
  }
  // Rows per CTA: 8 for one- to eight-row calls and for every gather call
  // (whose rows can carry different experts), 16 otherwise.
  const bool wide = a.rhs == nullptr && a.R > 8;
  if (xdt == kF16) return wide ? launch_mma<__half, 2>(a, st) : launch_mma<__half, 1>(a, st);
  return wide ? launch_mma<__nv_bfloat16, 2>(a, st) : launch_mma<__nv_bfloat16, 1>(a, st);
}

}  // namespace nvfp4
