// Decode-shape NVFP4 products: y[r, n] = factor(e_r) * sum_k x[lhs_r, k] * deq(w[e_r])[n, k].
//
// QuantizedMatmul below the tensor-core crossover and every GatherQMM decode
// (mlxcel PR #2629 "ROCm native NVFP4", Summary: the global scale is applied
// once per output; Changes during review: out-of-range expert rows are exact
// zeros).
//
// GB300 design. The work is bound by streaming the packed weights (9/16 byte
// per element). At HBM rate the SM has only about three instruction issues
// per weight element, so the decode must be lean and the multiply-add must not
// be SIMT: the weight fragment is decoded straight into registers in the
// m16n8k16 A-operand layout and the tokens ride in the 8-wide B operand.
//
//  * Thread-block clusters split K: the C CTAs of a cluster own the same 128
//    weight rows (a slab) and disjoint K slices. Each CTA stages its slice of
//    the activations in shared memory once and keeps it for every slab it
//    visits; partial sums are reduced across the cluster through distributed
//    shared memory (double-buffered per slab, one cluster barrier per slab),
//    so no global scratch memory is used.
//  * Decode precision. The fp4 * e4m3 product is exact in f16 and in bf16.
//    f16 decoding is two instructions per pair of elements (cvt + multiply);
//    bf16 needs four more. bf16 activations are therefore converted to f16
//    when staged, and the CTA checks that every staged element converts
//    exactly (a 16-bit range/precision check); if any does not, the CTA keeps
//    the bf16 values and decodes the weights to bf16 instead. Either way the
//    products entering the tensor core equal x * fp4 * e4m3 exactly and the
//    sum is accumulated in f32.
//  * K order inside one MMA is a permutation of the chunk's columns: in
//    k16-step s lane t's A slots {2t, 2t+1, 2t+8, 2t+9} hold columns
//    32t+4s+0..3 of its rows. A lane therefore streams four consecutive packed
//    words (one 128-bit load) per row and chunk, and the staged activations
//    are stored in the matching order so that its B operands for a chunk are
//    four conflict-free 128-bit shared loads.
#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

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
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Launch plan, computed on the host.
struct Plan {
  int C;            // cluster size = K split
  int nchunk;       // 128-column chunks in K
  int64_t slabs;    // 128-row slabs of N
  int spc;          // slabs per cluster (persistent loop)
  int TR;           // output rows (token slots) per CTA row tile
  int xs_stride;    // staged activation row stride in 16-bit elements
  int x_is_bf16;    // activation input is bf16 (else f16)
};

struct Chunk {
  uint4 wa, wb;     // words 4t..4t+3 of rows g and g+8
  uint32_t sa, sb;  // scale bytes of groups 2t, 2t+1 of rows g and g+8 (low 16 bits)
};

// Iterator over this warp's chunk jobs: slab-major, then expert pass, then chunk.
struct JobIter {
  int slab_i, pass, chunk;
  const uint32_t* pa;
  const uint32_t* pb;
  const uint8_t* qa;
  const uint8_t* qb;
  bool done;
};

struct Ctx {
  const uint32_t* w;
  const uint8_t* scales;
  int64_t N, kwords, kgroups;
  int64_t slab0, slab_step;  // first slab and stride between this cluster's slabs
  int nslab;                 // slabs this cluster visits
  int npass, cb, ce;
  const int* pass_e;
  int row_g;                 // warp*16 + g
};

__device__ __forceinline__ void iter_point(JobIter& it, const Ctx& c) {
  const int64_t slab = c.slab0 + (int64_t)it.slab_i * c.slab_step;
  const int64_t e = c.pass_e[it.pass];
  const int64_t na = slab * kSlabRows + c.row_g, nb = na + 8;
  const uint32_t* we = c.w + e * c.N * c.kwords;
  const uint8_t* se = c.scales + e * c.N * c.kgroups;
  it.pa = na < c.N ? we + na * c.kwords + (int64_t)it.chunk * 16 : nullptr;
  it.pb = nb < c.N ? we + nb * c.kwords + (int64_t)it.chunk * 16 : nullptr;
  it.qa = se + na * c.kgroups + (int64_t)it.chunk * 8;
  it.qb = se + nb * c.kgroups + (int64_t)it.chunk * 8;
}

__device__ __forceinline__ void iter_begin(JobIter& it, const Ctx& c) {
  it.slab_i = 0;
  it.pass = 0;
  it.chunk = c.cb;
  it.done = c.nslab <= 0 || c.cb >= c.ce || c.npass == 0;
  if (!it.done) iter_point(it, c);
}

// Advance; returns true when the job just left was the last of its slab.
__device__ __forceinline__ bool iter_next(JobIter& it, const Ctx& c) {
  if (++it.chunk < c.ce) {
    if (it.pa) it.pa += 16;
    if (it.pb) it.pb += 16;
    it.qa += 8;
    it.qb += 8;
    return false;
  }
  it.chunk = c.cb;
  bool slab_end = false;
  if (++it.pass >= c.npass) {
    it.pass = 0;
    slab_end = true;
    if (++it.slab_i >= c.nslab) {
      it.done = true;
      return true;
    }
  }
  iter_point(it, c);
  return slab_end;
}

template <bool VEC>
__device__ __forceinline__ void load_chunk(Chunk& ch, const JobIter& it, const Ctx& c, int t) {
  if (it.done) return;
  const int64_t kw = (int64_t)it.chunk * 16 + 4 * t;  // word index within the row
  if (VEC) {  // K % 32 == 0: a lane's four words (and two scales) are all in range or all out
    const bool ok = kw < c.kwords;
    ch.wa = (ok && it.pa) ? ld_stream_v4(it.pa + 4 * t) : make_uint4(0, 0, 0, 0);
    ch.wb = (ok && it.pb) ? ld_stream_v4(it.pb + 4 * t) : make_uint4(0, 0, 0, 0);
    ch.sa = (ok && it.pa) ? (uint32_t)__ldcs(reinterpret_cast<const unsigned short*>(it.qa + 2 * t)) : 0u;
    ch.sb = (ok && it.pb) ? (uint32_t)__ldcs(reinterpret_cast<const unsigned short*>(it.qb + 2 * t)) : 0u;
  } else {  // K % 32 == 16: words come in in-range pairs (one 16-column block each)
    const bool ok0 = kw < c.kwords, ok1 = kw + 2 < c.kwords;
    uint2 a0 = make_uint2(0, 0), a1 = a0, b0 = a0, b1 = a0;
    uint32_t sa = 0, sb = 0;
    if (it.pa) {
      if (ok0) { a0 = ld_stream_v2(it.pa + 4 * t); sa = it.qa[2 * t]; }
      if (ok1) { a1 = ld_stream_v2(it.pa + 4 * t + 2); sa |= (uint32_t)it.qa[2 * t + 1] << 8; }
    }
    if (it.pb) {
      if (ok0) { b0 = ld_stream_v2(it.pb + 4 * t); sb = it.qb[2 * t]; }
      if (ok1) { b1 = ld_stream_v2(it.pb + 4 * t + 2); sb |= (uint32_t)it.qb[2 * t + 1] << 8; }
    }
    ch.wa = make_uint4(a0.x, a0.y, a1.x, a1.y);
    ch.wb = make_uint4(b0.x, b0.y, b1.x, b1.y);
    ch.sa = sa;
    ch.sb = sb;
  }
}

__device__ __forceinline__ uint32_t u4get(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One chunk: decode eight words per lane and run 8 k16-steps per token tile.
// xaddr[mt] is the shared address of this lane's first staged activation
// group for the chunk (slot g+8mt), or 0 when the slot is not in the current
// pass. Column 32t+8q+i of a chunk is staged at offset (4q+t)*8+i, so the
// lane's q-th 16-byte group lies 64*q bytes after its base.
template <typename T, int MT>
__device__ __forceinline__ void compute_chunk(const Chunk& ch, const uint32_t (&xaddr)[MT], float (&acc)[MT][4]) {
  uint4 xv[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int q = 0; q < 4; ++q) xv[mt][q] = xaddr[mt] ? lds128(xaddr[mt] + 64 * q) : make_uint4(0, 0, 0, 0);
  const uint32_t sa0 = Dt<T>::scale(ch.sa & 0xFF), sa1 = Dt<T>::scale((ch.sa >> 8) & 0xFF);
  const uint32_t sb0 = Dt<T>::scale(ch.sb & 0xFF), sb1 = Dt<T>::scale((ch.sb >> 8) & 0xFF);
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // word j of the lane: columns 32t+8j..+7, k16-steps 2j and 2j+1
    uint32_t da[4], db[4];
    Dt<T>::decode(u4get(ch.wa, j), j < 2 ? sa0 : sa1, da);
    Dt<T>::decode(u4get(ch.wb, j), j < 2 ? sb0 : sb1, db);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int s = 2 * j + h;  // bytes 2h, 2h+1 of the word feed step s
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint32_t b0 = u4get(xv[mt][s >> 1], (2 * s) & 3);
        const uint32_t b1 = u4get(xv[mt][s >> 1], (2 * s + 1) & 3);
        MmaOp<T>::run(acc[mt], da[2 * h], db[2 * h], da[2 * h + 1], db[2 * h + 1], b0, b1);
      }
    }
  }
}

// Shared-memory layout (dynamic):
//   s_e[TR], s_xr[TR] (int64)      slot expert (-1 = zero row) and activation row
//   s_pe[TR] (int), s_pm[TR] (u32) expert and slot mask of each pass
//   xs[TR][xs_stride] (16-bit)     staged activations of this CTA's K slice
//   red[2][128][TR] (f32)          partial sums, double-buffered per slab
template <typename T, int MT, bool VEC>
__device__ __forceinline__ void run_slabs(const QmvArgs& a, const Plan& pl, const Ctx& c, uint32_t xs_base,
                                          uint32_t red_base, const int64_t* s_e, const uint32_t* s_pm,
                                          int64_t r0, uint32_t rank) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int TR = pl.TR;
  JobIter ld, cp;
  iter_begin(ld, c);
  iter_begin(cp, c);
  Chunk b0, b1, b2;
  load_chunk<VEC>(b0, ld, c, t);
  if (!ld.done) iter_next(ld, c);
  load_chunk<VEC>(b1, ld, c, t);
  if (!ld.done) iter_next(ld, c);

  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;
  int buf = 0;

  // staged activation address of this lane for chunk `chunk` of pass mask `pm`
  auto xaddrs = [&](uint32_t (&xa)[MT], int chunk, uint32_t pm) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int slot = g + 8 * mt;
      xa[mt] = (slot < TR && ((pm >> slot) & 1))
                   ? xs_base + 2u * (uint32_t)(slot * pl.xs_stride + (chunk - c.cb) * 128 + 8 * t) : 0u;
    }
  };
  // Per slab: partials -> shared, cluster barrier, reduce own rows over the cluster.
  auto flush = [&](int slab_i) {
    const uint32_t rb = red_base + (uint32_t)buf * (kSlabRows * TR * 4);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = warp * 16 + g + ((i & 2) ? 8 : 0);
        const int slot = 8 * mt + 2 * t + (i & 1);
        if (slot < TR) asm volatile("st.shared.f32 [%0], %1;" ::"r"(rb + 4u * (row * TR + slot)), "f"(acc[mt][i]));
        acc[mt][i] = 0.f;
      }
    cluster_arrive();
    cluster_wait();
    const int64_t slab = c.slab0 + (int64_t)slab_i * c.slab_step;
    const int rlo = (int)(rank * kSlabRows / pl.C), rhi = (int)((rank + 1) * kSlabRows / pl.C);
    const int nrow = rhi - rlo;
    for (int idx = threadIdx.x; idx < nrow * TR; idx += kThreads) {
      const int slot = idx / nrow, row = rlo + idx % nrow;
      const int64_t n = slab * kSlabRows + row, r = r0 + slot;
      if (n >= a.N || r >= a.R) continue;
      float v = 0.f;
      const uint32_t off = rb + 4u * (row * TR + slot);
      for (int q = 0; q < pl.C; ++q) v += ld_dsmem(map_rank(off, (uint32_t)q));
      const int64_t e = s_e[slot];
      const float out = e < 0 ? 0.f : (a.gs ? __fmul_rn(v, global_factor(a.gs, e)) : v);
      // the output has the activation input's dtype, whatever the MMA used
      if (pl.x_is_bf16)
        static_cast<__nv_bfloat16*>(a.y)[r * a.N + n] = __float2bfloat16_rn(out);
      else
        static_cast<__half*>(a.y)[r * a.N + n] = __float2half_rn(out);
    }
    buf ^= 1;
  };

  if (cp.done) {  // no weight to read (all rows zero): write the zero rows, join the barriers
    for (int s = 0; s < c.nslab; ++s) flush(s);
    return;
  }
  while (true) {
    // three register stages: two chunks in flight while one is decoded
    {
      load_chunk<VEC>(b2, ld, c, t);
      if (!ld.done) iter_next(ld, c);
      uint32_t xa[MT];
      xaddrs(xa, cp.chunk, s_pm[cp.pass]);
      compute_chunk<T, MT>(b0, xa, acc);
      const int si = cp.slab_i;
      if (iter_next(cp, c)) flush(si);
      if (cp.done) break;
    }
    {
      load_chunk<VEC>(b0, ld, c, t);
      if (!ld.done) iter_next(ld, c);
      uint32_t xa[MT];
      xaddrs(xa, cp.chunk, s_pm[cp.pass]);
      compute_chunk<T, MT>(b1, xa, acc);
      const int si = cp.slab_i;
      if (iter_next(cp, c)) flush(si);
      if (cp.done) break;
    }
    {
      load_chunk<VEC>(b1, ld, c, t);
      if (!ld.done) iter_next(ld, c);
      uint32_t xa[MT];
      xaddrs(xa, cp.chunk, s_pm[cp.pass]);
      compute_chunk<T, MT>(b2, xa, acc);
      const int si = cp.slab_i;
      if (iter_next(cp, c)) flush(si);
      if (cp.done) break;
    }
  }
}

template <int MT, bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
qmv_cluster_kernel(const QmvArgs a, const Plan pl) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int TR = pl.TR;
  int64_t* s_e = reinterpret_cast<int64_t*>(smem);
  int64_t* s_xr = s_e + TR;
  int* s_pe = reinterpret_cast<int*>(s_xr + TR);
  uint32_t* s_pm = reinterpret_cast<uint32_t*>(s_pe + TR);
  __shared__ int s_npass;
  const size_t meta = ((size_t)TR * 24 + 15) & ~(size_t)15;
  uint8_t* xs = smem + meta;
  const size_t xs_bytes = (size_t)TR * pl.xs_stride * 2;
  const uint32_t xs_base = (uint32_t)__cvta_generic_to_shared(xs);
  const uint32_t red_base = xs_base + (uint32_t)((xs_bytes + 15) & ~(size_t)15);

  const uint32_t rank = cluster_rank();
  const int64_t cluster_id = blockIdx.x / pl.C;
  const int64_t nclusters = gridDim.x / pl.C;
  const int64_t r0 = (int64_t)blockIdx.y * TR;

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
    s_npass = np;  // 0 when every row of the tile is a zero row: no weight is read
  }

  // This CTA's K slice.
  const int cb = (int)((int64_t)pl.nchunk * rank / pl.C), ce = (int)((int64_t)pl.nchunk * (rank + 1) / pl.C);
  // Stage activations of the slice: element at column 32t+8q+i of a chunk is
  // stored at chunk offset (4q+t)*8+i so a lane's four 16-byte reads are
  // contiguous with its neighbours'.
  const int units = TR * (ce - cb) * 16;  // 8-element units
  int inexact = 0;
  for (int u = threadIdx.x; u < units; u += kThreads) {
    const int slot = u / ((ce - cb) * 16);
    const int rem = u % ((ce - cb) * 16);
    const int ch = rem >> 4, w8 = rem & 15;  // unit within chunk: columns 8*w8 .. 8*w8+7
    const int tq = w8 >> 2, qq = w8 & 3;     // t = w8/4, q = w8%4
    const int64_t col = (int64_t)(cb + ch) * 128 + 8 * w8;
    const int64_t xr = s_xr[slot];
    uint4 v = make_uint4(0, 0, 0, 0);
    if (s_e[slot] >= 0 && col < a.K)
      v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + xr * a.K + col));
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
    const uint32_t dst = xs_base + 2u * (uint32_t)(slot * pl.xs_stride + ch * 128 + (4 * qq + tq) * 8);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
  }
  const bool use_bf16 = __syncthreads_or(inexact) != 0;
  if (use_bf16) {  // keep the exact bf16 activations instead
    for (int u = threadIdx.x; u < units; u += kThreads) {
      const int slot = u / ((ce - cb) * 16);
      const int rem = u % ((ce - cb) * 16);
      const int ch = rem >> 4, w8 = rem & 15, tq = w8 >> 2, qq = w8 & 3;
      const int64_t col = (int64_t)(cb + ch) * 128 + 8 * w8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (s_e[slot] >= 0 && col < a.K)
        v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + s_xr[slot] * a.K + col));
      const uint32_t dst = xs_base + 2u * (uint32_t)(slot * pl.xs_stride + ch * 128 + (4 * qq + tq) * 8);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
    }
    __syncthreads();
  }

  Ctx c;
  c.w = a.w;
  c.scales = a.scales;
  c.N = a.N;
  c.kwords = a.K / 8;
  c.kgroups = a.K / 16;
  c.slab0 = cluster_id;
  c.slab_step = nclusters;
  c.nslab = (int)(cluster_id < pl.slabs ? (pl.slabs - cluster_id + nclusters - 1) / nclusters : 0);
  c.npass = s_npass;
  c.cb = cb;
  c.ce = ce;
  c.pass_e = s_pe;
  c.row_g = (threadIdx.x >> 5) * 16 + ((threadIdx.x & 31) >> 2);
  if (use_bf16)
    run_slabs<__nv_bfloat16, MT, VEC>(a, pl, c, xs_base, red_base, s_e, s_pm, r0, rank);
  else
    run_slabs<__half, MT, VEC>(a, pl, c, xs_base, red_base, s_e, s_pm, r0, rank);
  // Peers may still read this CTA's partials: leave together.
  cluster_arrive();
  cluster_wait();
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

int sm_count() {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

constexpr size_t kSmemBudget = 110 * 1024;  // two CTAs per SM

size_t smem_bytes(const Plan& p) {
  const size_t meta = ((size_t)p.TR * 24 + 15) & ~(size_t)15;
  const size_t xs = (((size_t)p.TR * p.xs_stride * 2) + 15) & ~(size_t)15;
  const size_t red = (size_t)2 * kSlabRows * p.TR * 4;
  return meta + xs + red;
}

template <int MT>
cudaError_t launch_cluster(const QmvArgs& a, Plan pl, cudaStream_t st) {
  pl.TR = 8 * MT;
  const int64_t row_tiles = (a.R + pl.TR - 1) / pl.TR;
  // K split: a divisor of the chunk count up to 8 when one exists, at least
  // four chunks per CTA.
  int C = 1;
  for (int c = 8; c >= 1; --c) {
    if (pl.nchunk >= 4 * c && pl.nchunk % c == 0) { C = c; break; }
  }
  if (C == 1 && pl.nchunk >= 16) C = 8;
  pl.C = C;
  const int max_slice = (pl.nchunk + C - 1) / C;
  // staged row stride: 128-byte multiple plus 64 bytes (conflict-free LDS.128)
  pl.xs_stride = max_slice * 128 + 32;
  // persistent clusters: enough CTAs to fill the GPU twice, slabs spread evenly
  const int64_t cap = (int64_t)sm_count() * 2;
  const int64_t want_clusters = cap / (C * row_tiles) > 0 ? cap / (C * row_tiles) : 1;
  int64_t spc = (pl.slabs + want_clusters - 1) / want_clusters;
  if (spc < 1) spc = 1;
  const int64_t nclusters = (pl.slabs + spc - 1) / spc;
  pl.spc = (int)spc;
  const size_t smem = smem_bytes(pl);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;  // excluded by qmv_supported_k
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nclusters * C), (unsigned)row_tiles, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (a.K % 32 == 0) {
    e = cudaFuncSetAttribute(qmv_cluster_kernel<MT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, qmv_cluster_kernel<MT, true>, a, pl);
  }
  e = cudaFuncSetAttribute(qmv_cluster_kernel<MT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, qmv_cluster_kernel<MT, false>, a, pl);
}

}  // namespace

cudaError_t launch_qmv(const QmvArgs& a, int xdt, cudaStream_t st) {
  if (xdt == kF32) {
    const dim3 grid((unsigned)((a.N + kWarps - 1) / kWarps), (unsigned)((a.R + kF32Tokens - 1) / kF32Tokens));
    qmv_f32_kernel<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
  }
  Plan pl{};
  pl.nchunk = (int)((a.K + 127) / 128);
  pl.slabs = (a.N + kSlabRows - 1) / kSlabRows;
  pl.x_is_bf16 = xdt == kBF16;
  // Rows per CTA tile: 8 for one- to eight-row calls and for gather calls,
  // 16 otherwise, unless the staged slice would not fit.
  const bool wide = a.rhs == nullptr && a.R > 8;
  Plan probe = pl;
  probe.TR = 16;
  probe.xs_stride = ((pl.nchunk + 7) / 8) * 128 + 32;
  if (wide && smem_bytes(probe) <= kSmemBudget) return launch_cluster<2>(a, pl, st);
  return launch_cluster<1>(a, pl, st);
}

bool qmv_supported_k(int64_t K) { return K <= kQmvMaxK; }

}  // namespace nvfp4
