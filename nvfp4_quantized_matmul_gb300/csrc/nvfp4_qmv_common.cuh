// Shared pieces of the decode-shape kernels (csrc/nvfp4_qmv.cu and
// csrc/nvfp4_qmv_tma.cu): tiling constants, the m16n8k16 MMA wrappers,
// cluster/DSMEM helpers, the per-chunk decode + MMA step and the staging of
// the activation slice.
#pragma once
#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace qmv {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlabRows = kWarps * 16;  // 128 weight rows per slab

template <typename T> struct MmaOp;
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

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
// Arrival that publishes nothing (a warp whose writes no peer reads): it does
// not wait for the thread's outstanding memory operations.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Cluster reduction of one slab, split in two so that the output stores can
// be issued after the next cluster arrive (a release fence would otherwise
// wait for them). This CTA (rank `rank` of C) owns rows [rank*128/C,
// (rank+1)*128/C) of the slab; partial sums sit at rb + 4*(row*TR + slot) in
// every CTA of the cluster. An item is one row and four consecutive slots; a
// thread holds at most two items (nrow * TR/4 <= 512 for 256 threads). All
// remote 16-byte loads of a group of four peers are issued before any is
// summed, so the distributed-shared-memory latency is paid once per group.
struct ReduceOut {
  float v[2][4];
  int n;
};
static __device__ __noinline__ void cluster_gather(int C, int TR, uint32_t rank, uint32_t rb, int tid, int nthreads,
                                                   ReduceOut& o) {
  const int rlo = (int)(rank * kSlabRows / C), rhi = (int)((rank + 1) * kSlabRows / C);
  const int nrow = rhi - rlo, nq = TR / 4;
  o.n = 0;
  for (int idx = tid, k = 0; idx < nrow * nq && k < 2; idx += nthreads, ++k) {
    const int quad = idx / nrow, row = rlo + idx % nrow;
    const uint32_t off = rb + 4u * (uint32_t)(row * TR + 4 * quad);
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    for (int q0 = 0; q0 < C; q0 += 4) {
      float4 part[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q0 + q < C) part[q] = ld_dsmem4(map_rank(off, (uint32_t)(q0 + q)));
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q0 + q < C) {
          v[0] += part[q].x;
          v[1] += part[q].y;
          v[2] += part[q].z;
          v[3] += part[q].w;
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) o.v[k][j] = v[j];
    o.n = k + 1;
  }
}
// Writes factor * sum (or +0.0 for zero rows) in the activation dtype.
static __device__ __noinline__ void cluster_store(const QmvArgs& a, int C, int TR, int x_is_bf16, uint32_t rank,
                                                  int64_t slab, const int64_t* s_e, int64_t r0, int tid, int nthreads,
                                                  const ReduceOut& o) {
  const int rlo = (int)(rank * kSlabRows / C), rhi = (int)((rank + 1) * kSlabRows / C);
  const int nrow = rhi - rlo;
  for (int k = 0; k < o.n; ++k) {
    const int idx = tid + k * nthreads;
    const int quad = idx / nrow, row = rlo + idx % nrow;
    const int64_t n = slab * kSlabRows + row;
    if (n >= a.N) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int slot = 4 * quad + j;
      const int64_t r = r0 + slot;
      if (r >= a.R) continue;
      const int64_t e = s_e[slot];
      const float out = e < 0 ? 0.f : (a.gs ? __fmul_rn(o.v[k][j], global_factor(a.gs, e)) : o.v[k][j]);
      // the output has the activation input's dtype, whatever the MMA used
      if (x_is_bf16)
        static_cast<__nv_bfloat16*>(a.y)[r * a.N + n] = __float2bfloat16_rn(out);
      else
        static_cast<__half*>(a.y)[r * a.N + n] = __float2half_rn(out);
    }
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}


constexpr int kChunkCols = 256;  // columns per job: 32 packed words per row
constexpr int kChunkWords = kChunkCols / 8;

// Launch plan, computed on the host.
struct Plan {
  int C;            // cluster size = K split
  int nchunk;       // 256-column chunks in K
  int64_t slabs;    // 128-row slabs of N
  int spc;          // slabs per cluster (persistent loop)
  int TR;           // output rows (token slots) per CTA row tile
  int xs_stride;    // staged activation row stride in 16-bit elements
  int x_is_bf16;    // activation input is bf16 (else f16)
  int stages;       // depth of the TMA stage ring (TMA-fed kernel only)
  int xs_slots;     // staged activation rows actually allocated (min(TR, R))
};

// One lane's share of a chunk: words 8t..8t+7 of rows g and g+8, and the
// four scale bytes (groups 4t..4t+3) of each row.
struct Chunk {
  uint4 a0, a1, b0, b1;
  uint32_t sa, sb;
};

__device__ __forceinline__ uint32_t u4get(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Block-scale operand for word j of a row: the f16 path converts the E4M3
// byte directly (two instructions); the bf16 path reads scale * 2^112 from a
// 256-entry table built once per CTA.
template <typename T> __device__ __forceinline__ uint32_t scale_op(uint32_t sbytes, int grp, uint32_t lut_bf);
template <> __device__ __forceinline__ uint32_t scale_op<__half>(uint32_t sbytes, int grp, uint32_t) {
  return e4m3_to_f16x2_bcast(sbytes >> (8 * grp));
}
template <> __device__ __forceinline__ uint32_t scale_op<__nv_bfloat16>(uint32_t sbytes, int grp, uint32_t lut_bf) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(lut_bf + 4u * ((sbytes >> (8 * grp)) & 0xFFu)));
  return v;
}

// Block-scale operands for the two 16-column groups of one half-chunk
// (scale bytes 2*half and 2*half+1 of the lane's scale word), each broadcast
// to both halves of a packed register. f16: one two-byte conversion and two
// byte permutes; bf16: two lookups of scale * 2^112 in the shared table.
template <typename T>
__device__ __forceinline__ void scale_pair(uint32_t sbytes, int half, uint32_t lut_bf, uint32_t& s0, uint32_t& s1);
template <>
__device__ __forceinline__ void scale_pair<__half>(uint32_t sbytes, int half, uint32_t, uint32_t& s0, uint32_t& s1) {
  const uint32_t h = e4m3x2_to_f16x2(sbytes >> (16 * half));
  s0 = __byte_perm(h, 0, 0x1010);
  s1 = __byte_perm(h, 0, 0x3232);
}
template <>
__device__ __forceinline__ void scale_pair<__nv_bfloat16>(uint32_t sbytes, int half, uint32_t lut_bf, uint32_t& s0,
                                                          uint32_t& s1) {
  s0 = scale_op<__nv_bfloat16>(sbytes, 2 * half, lut_bf);
  s1 = scale_op<__nv_bfloat16>(sbytes, 2 * half + 1, lut_bf);
}

// One chunk: 16 k16-steps. Lane t's word j holds columns 64t+8j..+7; step s
// uses bytes 2h, 2h+1 (h = s & 1) of word s/2, i.e. columns 64t+4s+0..3 in
// A slots {2t, 2t+1, 2t+8, 2t+9}. The staged activations put column
// 64t+8q+i of the chunk at offset (4q+t)*8+i, so the lane's q-th 16-byte group
// lies 64*q bytes after its base (8t elements into the chunk).
// Accumulator sets: consecutive k-steps rotate over NACC independent sets so
// the MMAs of a chunk form NACC dependency chains instead of one (summed when
// the slab is flushed).
template <int MT> struct NAcc { static constexpr int value = MT == 1 ? 4 : 2; };

template <typename T, int MT>
__device__ __forceinline__ void compute_chunk(const Chunk& ch, const uint32_t (&xaddr)[MT],
                                              float (&acc)[NAcc<MT>::value][MT][4], uint32_t lut_bf) {
  constexpr int NA = NAcc<MT>::value;
#pragma unroll
  for (int half = 0; half < 2; ++half) {  // words 4*half .. 4*half+3
    // xaddr points at a zeroed block for slots outside the pass, so the
    // loads are unconditional
    uint4 xv[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[mt][q] = lds128(xaddr[mt] + 64 * (4 * half + q));
    const uint4& wa = half ? ch.a1 : ch.a0;
    const uint4& wb = half ? ch.b1 : ch.b0;
    uint32_t sa0, sa1, sb0, sb1;
    scale_pair<T>(ch.sa, half, lut_bf, sa0, sa1);
    scale_pair<T>(ch.sb, half, lut_bf, sb0, sb1);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t da[4], db[4];
      Dt<T>::decode(u4get(wa, j), j < 2 ? sa0 : sa1, da);
      Dt<T>::decode(u4get(wb, j), j < 2 ? sb0 : sb1, db);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int sl = 2 * j + h;  // step within this half: x group sl/2, u32 pair (sl&1)*2
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t b0 = u4get(xv[mt][sl >> 1], 2 * (sl & 1));
          const uint32_t b1 = u4get(xv[mt][sl >> 1], 2 * (sl & 1) + 1);
          MmaOp<T>::run(acc[(8 * half + sl) % NA][mt], da[2 * h], db[2 * h], da[2 * h + 1], db[2 * h + 1], b0, b1);
        }
      }
    }
  }
}


// Slot metadata of the CTA's row tile: expert (-1 = zero row) and activation
// row per slot, then one pass per distinct expert (thread 0). Ends with the
// pass table visible to the block.
__device__ __forceinline__ void setup_slots(const QmvArgs& a, int TR, int64_t r0, int64_t* s_e, int64_t* s_xr,
                                            int* s_pe, uint32_t* s_pm, int* s_npass) {
  if (threadIdx.x < TR) {
    const int64_t r = r0 + threadIdx.x;
    int64_t e = -1, xr = -1;
    if (r < a.R) {
      e = a.rhs ? (int64_t)a.rhs[r] : 0;
      xr = a.lhs ? (int64_t)a.lhs[r] : r;
      if (e >= a.E || xr >= a.B) e = -1;  // zero row
    }
    s_e[threadIdx.x] = e;
    s_xr[threadIdx.x] = xr;
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // group the slots by expert: one pass per distinct expert
    uint32_t pending = 0;
    for (int j = 0; j < TR; ++j)
      if (s_e[j] >= 0) pending |= 1u << j;
    int np = 0;
    while (pending) {
      const int first = __ffs(pending) - 1;
      const int64_t e = s_e[first];
      uint32_t m = 0;
      for (int j = first; j < TR; ++j)
        if (((pending >> j) & 1) && s_e[j] == e) m |= 1u << j;
      pending &= ~m;
      s_pe[np] = (int)e;
      s_pm[np] = m;
      ++np;
    }
    *s_npass = np;  // 0 when every row of the tile is a zero row: no weight is read
  }

  __syncthreads();
}

// Stage this CTA's slice of the activations (chunks cb..ce-1 of every slot)
// in 8-element units: column 64t+8q+i of a chunk goes to chunk offset
// (4q+t)*8+i. bf16 inputs are converted to f16 when every staged element
// converts exactly; otherwise the bf16 values are staged. Returns true (for
// the whole block) when the staged values are bf16.
__device__ __forceinline__ bool stage_x(const QmvArgs& a, const Plan& pl, int cb, int ce, uint32_t xs_base,
                                        const int64_t* s_e, const int64_t* s_xr) {
  const int TR = pl.TR;
  const int upc = kChunkCols / 8;  // units per chunk and slot
  const int units = TR * (ce - cb) * upc;
  int inexact = 0;
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    const int slot = u / ((ce - cb) * upc);
    const int rem = u % ((ce - cb) * upc);
    const int ch = rem / upc, w8 = rem % upc;  // columns 8*w8 .. 8*w8+7 of the chunk
    const int tq = w8 >> 3, qq = w8 & 7;
    const int64_t col = (int64_t)(cb + ch) * kChunkCols + 8 * w8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (s_e[slot] >= 0 && col < a.K)
      v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + s_xr[slot] * a.K + col));
    if (pl.x_is_bf16) {  // bf16 -> f16, exactness checked
      uint32_t in[4] = {v.x, v.y, v.z, v.w}, o[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float lo = __uint_as_float(in[p] << 16), hi = __uint_as_float(in[p] & 0xFFFF0000u);
        const __half2 h = __floats2half2_rn(lo, hi);
        const float2 back = __half22float2(h);
        inexact |= (back.x != lo) | (back.y != hi);
        o[p] = *reinterpret_cast<const uint32_t*>(&h);
      }
      v = make_uint4(o[0], o[1], o[2], o[3]);
    }
    const uint32_t dst = xs_base + 2u * (uint32_t)(slot * pl.xs_stride + ch * kChunkCols + (4 * qq + tq) * 8);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
  }
  const bool use_bf16 = __syncthreads_or(inexact) != 0;
  if (use_bf16) {  // keep the exact bf16 activations instead
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
      const int slot = u / ((ce - cb) * upc);
      const int rem = u % ((ce - cb) * upc);
      const int ch = rem / upc, w8 = rem % upc, tq = w8 >> 3, qq = w8 & 7;
      const int64_t col = (int64_t)(cb + ch) * kChunkCols + 8 * w8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (s_e[slot] >= 0 && col < a.K)
        v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + s_xr[slot] * a.K + col));
      const uint32_t dst = xs_base + 2u * (uint32_t)(slot * pl.xs_stride + ch * kChunkCols + (4 * qq + tq) * 8);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
    }
    __syncthreads();
  }

  return use_bf16;
}

// Synchronisation of the staging threads: named barrier 1 over kCount
// threads (the staging group), with an OR-reduction variant.
template <int kCount>
__device__ __forceinline__ int sync_or(int pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbarrier.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(kCount)
      : "memory");
  return (int)r;
}
template <int kCount>
__device__ __forceinline__ void sync_all() {
  asm volatile("barrier.sync 1, %0;" ::"n"(kCount) : "memory");
}

// Exact residual of one staged activation that f16 cannot hold (a bf16 value
// below the f16 normal range with more significant bits than f16 keeps
// there): the f16 fast path adds fp4 * e4m3 * r in f32 for it.
struct Corr {
  int slot;  // token slot
  int col;   // column within this CTA's K slice
  float r;   // x - f16(x), exact in f32
};
constexpr int kMaxCorr = 64;

// stage_x with residual corrections: returns 0 (f16, exact), 1 (f16 plus the
// `*n_corr` corrections, sorted by column) or 2 (bf16 staged: some value
// overflows f16 or is NaN, or more than kMaxCorr values need a residual).
// `*n_corr` must be zero on entry (and visible to the block).
// Threads kFirst .. kFirst+kCount-1 (whole warps) take part.
// dst(slot, ch, w8) gives the shared address of the 16-byte unit holding
// columns 8*w8 .. 8*w8+7 of chunk ch (relative to the slice) of a slot.
template <int kFirst, int kCount, typename Dst>
__device__ __forceinline__ int stage_x_corr(const QmvArgs& a, const Plan& pl, int cb, int ce, Dst dst_of,
                                            const int64_t* s_e, const int64_t* s_xr, Corr* corr, int* n_corr) {
  // only the allocated slots (min(TR, R)) are staged; the others never hold
  // a row of this tile and are never read
  const int upc = kChunkCols / 8;
  const int units = pl.xs_slots * (ce - cb) * upc;
  const int nthr = kCount, tid = (int)threadIdx.x - kFirst;
  int hard = 0;
  for (int u = tid; u < units; u += nthr) {
    const int slot = u / ((ce - cb) * upc);
    const int rem = u % ((ce - cb) * upc);
    const int ch = rem / upc, w8 = rem % upc;
    const int64_t col = (int64_t)(cb + ch) * kChunkCols + 8 * w8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (s_e[slot] >= 0 && col < a.K)
      v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + s_xr[slot] * a.K + col));
    if (pl.x_is_bf16) {
      uint32_t in[4] = {v.x, v.y, v.z, v.w}, o[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float lo = __uint_as_float(in[p] << 16), hi = __uint_as_float(in[p] & 0xFFFF0000u);
        const __half2 h = __floats2half2_rn(lo, hi);
        const float2 back = __half22float2(h);
        o[p] = *reinterpret_cast<const uint32_t*>(&h);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float xv = e ? hi : lo, bv = e ? back.y : back.x;
          if (bv != xv) {
            if (!(fabsf(xv) <= 65504.f)) {  // overflow or NaN: no f16 + residual split
              hard = 1;
            } else {
              const int i = atomicAdd(n_corr, 1);
              if (i < kMaxCorr) corr[i] = Corr{slot, ch * kChunkCols + 8 * w8 + 2 * p + e, xv - bv};
              else hard = 1;
            }
          }
        }
      }
      v = make_uint4(o[0], o[1], o[2], o[3]);
    }
    const uint32_t dst = dst_of(slot, ch, w8);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
  }
  if (sync_or<kCount>(hard)) {  // keep the exact bf16 activations instead
    for (int u = tid; u < units; u += nthr) {
      const int slot = u / ((ce - cb) * upc);
      const int rem = u % ((ce - cb) * upc);
      const int ch = rem / upc, w8 = rem % upc;
      const int64_t col = (int64_t)(cb + ch) * kChunkCols + 8 * w8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (s_e[slot] >= 0 && col < a.K)
        v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + s_xr[slot] * a.K + col));
      const uint32_t dst = dst_of(slot, ch, w8);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
    }
    sync_all<kCount>();
    return 2;
  }
  const int nc = *n_corr;
  if (nc == 0) return 0;
  if (tid == 0) {  // sort by column (at most kMaxCorr entries)
    for (int i = 1; i < nc; ++i) {
      const Corr k = corr[i];
      int j = i - 1;
      while (j >= 0 && corr[j].col > k.col) {
        corr[j + 1] = corr[j];
        --j;
      }
      corr[j + 1] = k;
    }
  }
  sync_all<kCount>();
  return 1;
}

// Value of one E2M1 code as float (exact): magnitude 2^(e-1) * (1 + m/2) for
// exponent bits e > 0, m/2 for e = 0; bit 3 is the sign.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  const uint32_t e = (c >> 1) & 3, m = c & 1;
  const uint32_t bits = e ? ((e + 126u) << 23) | (m << 22) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(bits | ((c & 8u) << 28));
}

}  // namespace qmv
}  // namespace nvfp4
