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
//  * K order inside one MMA is a permutation of the chunk's columns: with
//    256-column chunks, in k16-step s lane t's A slots {2t, 2t+1, 2t+8, 2t+9}
//    hold columns 64t+4s+0..3 of its rows. A lane therefore streams eight
//    consecutive packed words (two 128-bit loads) per row and chunk, and the
//    staged activations are stored in the matching order so that its B
//    operands are conflict-free 128-bit shared loads.
#include "nvfp4_qmv_common.cuh"

namespace nvfp4 {
namespace {
using namespace qmv;

// Load-side iterator over this warp's jobs: slab-major, then expert pass,
// then chunk. Only the loads need addresses; the compute side counts.
struct LoadIter {
  int slab_i, pass, chunk;
  const uint32_t* pa;  // row n0+g of the current expert, at the chunk (null if n >= N)
  const uint32_t* pb;  // row n0+g+8
  const uint8_t* qa;
  const uint8_t* qb;
  bool done;
};
struct CountIter {
  int slab_i, pass, chunk;
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

__device__ __forceinline__ void iter_point(LoadIter& it, const Ctx& c) {
  const int64_t slab = c.slab0 + (int64_t)it.slab_i * c.slab_step;
  const int64_t e = c.pass_e[it.pass];
  const int64_t na = slab * kSlabRows + c.row_g, nb = na + 8;
  const uint32_t* we = c.w + e * c.N * c.kwords;
  const uint8_t* se = c.scales + e * c.N * c.kgroups;
  const int64_t kw = (int64_t)it.chunk * kChunkWords, kg = (int64_t)it.chunk * (kChunkCols / 16);
  it.pa = na < c.N ? we + na * c.kwords + kw : nullptr;
  it.pb = nb < c.N ? we + nb * c.kwords + kw : nullptr;
  it.qa = se + na * c.kgroups + kg;
  it.qb = se + nb * c.kgroups + kg;
}

template <typename It>
__device__ __forceinline__ bool empty_job_list(const Ctx& c) {
  return c.nslab <= 0 || c.cb >= c.ce || c.npass == 0;
}

__device__ __forceinline__ void iter_begin(LoadIter& it, const Ctx& c) {
  it.slab_i = 0;
  it.pass = 0;
  it.chunk = c.cb;
  it.done = empty_job_list<LoadIter>(c);
  if (!it.done) iter_point(it, c);
}
__device__ __forceinline__ void iter_begin(CountIter& it, const Ctx& c) {
  it.slab_i = 0;
  it.pass = 0;
  it.chunk = c.cb;
  it.done = empty_job_list<CountIter>(c);
}

__device__ __forceinline__ void iter_next(LoadIter& it, const Ctx& c) {
  if (++it.chunk < c.ce) {
    if (it.pa) it.pa += kChunkWords;
    if (it.pb) it.pb += kChunkWords;
    it.qa += kChunkCols / 16;
    it.qb += kChunkCols / 16;
    return;
  }
  it.chunk = c.cb;
  if (++it.pass >= c.npass) {
    it.pass = 0;
    if (++it.slab_i >= c.nslab) {
      it.done = true;
      return;
    }
  }
  iter_point(it, c);
}
// Advance; returns true when the job just left was the last of its slab.
__device__ __forceinline__ bool iter_next(CountIter& it, const Ctx& c) {
  if (++it.chunk < c.ce) return false;
  it.chunk = c.cb;
  if (++it.pass < c.npass) return false;
  it.pass = 0;
  if (++it.slab_i >= c.nslab) it.done = true;
  return true;
}

// KV = 2: K % 64 == 0 (two 128-bit loads and one 32-bit scale load per row);
// KV = 1: K % 32 == 0 (scales as two 16-bit halves); KV = 0: K % 16 == 0
// (words in 64-bit pairs, scales bytewise).
template <int KV>
__device__ __forceinline__ void load_row(const uint32_t* p, const uint8_t* q, int64_t kw0, int64_t kwords, int t,
                                         uint4& lo, uint4& hi, uint32_t& sc) {
  lo = make_uint4(0, 0, 0, 0);
  hi = lo;
  sc = 0;
  if (!p) return;
  if (KV >= 1) {
    const bool ok0 = kw0 < kwords, ok1 = kw0 + 4 < kwords;
    if (ok0) lo = ld_stream_v4(p + 8 * t);
    if (ok1) hi = ld_stream_v4(p + 8 * t + 4);
    if (KV == 2) {
      if (ok1) sc = __ldcs(reinterpret_cast<const unsigned int*>(q + 4 * t));
      else if (ok0) sc = __ldcs(reinterpret_cast<const unsigned short*>(q + 4 * t));
    } else {
      if (ok0) sc = __ldcs(reinterpret_cast<const unsigned short*>(q + 4 * t));
      if (ok1) sc |= (uint32_t)__ldcs(reinterpret_cast<const unsigned short*>(q + 4 * t + 2)) << 16;
    }
  } else {
    uint32_t wv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      if (kw0 + 2 * pr < kwords) {
        const uint2 v = ld_stream_v2(p + 8 * t + 2 * pr);
        wv[2 * pr] = v.x;
        wv[2 * pr + 1] = v.y;
        sc |= (uint32_t)q[4 * t + pr] << (8 * pr);
      }
    }
    lo = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    hi = make_uint4(wv[4], wv[5], wv[6], wv[7]);
  }
}

template <int KV>
__device__ __forceinline__ void load_chunk(Chunk& ch, const LoadIter& it, const Ctx& c, int t) {
  if (it.done) return;
  const int64_t kw0 = (int64_t)it.chunk * kChunkWords + 8 * t;
  load_row<KV>(it.pa, it.qa, kw0, c.kwords, t, ch.a0, ch.a1, ch.sa);
  load_row<KV>(it.pb, it.qb, kw0, c.kwords, t, ch.b0, ch.b1, ch.sb);
}

// Shared-memory layout (dynamic):
//   s_e[TR], s_xr[TR] (int64)      slot expert (-1 = zero row) and activation row
//   s_pe[TR] (int), s_pm[TR] (u32) expert and slot mask of each pass
//   lut_bf[256] (u32)              bf16x2 of scale * 2^112 per E4M3 byte
//   xs[TR][xs_stride] (16-bit)     staged activations of this CTA's K slice
//   red[2][128][TR] (f32)          partial sums, double-buffered per slab
template <typename T, int MT, int KV>
__device__ __forceinline__ void run_slabs(const QmvArgs& a, const Plan& pl, const Ctx& c, uint32_t xs_base,
                                          uint32_t red_base, uint32_t lut_bf, uint32_t zero_base, const int64_t* s_e,
                                          const uint32_t* s_pm, int64_t r0, uint32_t rank) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int TR = pl.TR;
  LoadIter ld;
  CountIter cp;
  iter_begin(ld, c);
  iter_begin(cp, c);
  Chunk b0, b1;
  load_chunk<KV>(b0, ld, c, t);
  if (!ld.done) iter_next(ld, c);

  constexpr int NA = NAcc<MT>::value;
  float acc[NA][MT][4];
#pragma unroll
  for (int k = 0; k < NA; ++k)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[k][mt][i] = 0.f;
  int buf = 0;
  int pending = -1;  // slab whose cluster reduction is still to do

  auto xaddrs = [&](uint32_t (&xa)[MT], int chunk, uint32_t pm) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int slot = g + 8 * mt;
      xa[mt] = (slot < TR && ((pm >> slot) & 1))
                   ? xs_base + 2u * (uint32_t)(slot * pl.xs_stride + (chunk - c.cb) * kChunkCols + 8 * t)
                   : zero_base + 16u * (uint32_t)t;
    }
  };
  // Sum slab `si`'s partials (buffer `rb`) over the cluster for this CTA's rows.
  ReduceOut red_out;
  auto gather = [&](uint32_t rb) { cluster_gather(pl.C, TR, rank, rb, threadIdx.x, kThreads, red_out); };
  auto store = [&](int si) {
    cluster_store(a, pl.C, TR, pl.x_is_bf16, rank, c.slab0 + (int64_t)si * c.slab_step, s_e, r0, threadIdx.x,
                  kThreads, red_out);
  };
  const uint32_t buf_bytes = (uint32_t)(kSlabRows * TR * 4);
  // End of slab `si`: reduce the previous slab (one cluster barrier behind, so
  // no CTA waits for the others while it still has work), then publish this
  // slab's partials.
  auto flush = [&](int si) {
    if (pending >= 0) {
      cluster_wait();
      gather(red_base + (uint32_t)(buf ^ 1) * buf_bytes);
    }
    const uint32_t rb = red_base + (uint32_t)buf * buf_bytes;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = warp * 16 + g + ((i & 2) ? 8 : 0);
        const int slot = 8 * mt + 2 * t + (i & 1);
        float v = 0.f;
#pragma unroll
        for (int k = 0; k < NA; ++k) {
          v += acc[k][mt][i];
          acc[k][mt][i] = 0.f;
        }
        if (slot < TR) asm volatile("st.shared.f32 [%0], %1;" ::"r"(rb + 4u * (row * TR + slot)), "f"(v));
      }
    cluster_arrive();
    if (pending >= 0) store(pending);  // after the arrive: its release does not wait for these stores
    pending = si;
    buf ^= 1;
  };

  if (cp.done) {  // no weight to read (all rows zero): write the zero rows, join the barriers
    for (int s = 0; s < c.nslab; ++s) flush(s);
  } else {
    while (true) {  // two register stages: one chunk in flight while one is decoded
      {
        load_chunk<KV>(b1, ld, c, t);
        if (!ld.done) iter_next(ld, c);
        uint32_t xa[MT];
        xaddrs(xa, cp.chunk, s_pm[cp.pass]);
        compute_chunk<T, MT>(b0, xa, acc, lut_bf);
        const int si = cp.slab_i;
        if (iter_next(cp, c)) flush(si);
        if (cp.done) break;
      }
      {
        load_chunk<KV>(b0, ld, c, t);
        if (!ld.done) iter_next(ld, c);
        uint32_t xa[MT];
        xaddrs(xa, cp.chunk, s_pm[cp.pass]);
        compute_chunk<T, MT>(b1, xa, acc, lut_bf);
        const int si = cp.slab_i;
        if (iter_next(cp, c)) flush(si);
        if (cp.done) break;
      }
    }
  }
  if (pending >= 0) {
    cluster_wait();
    gather(red_base + (uint32_t)(buf ^ 1) * buf_bytes);
    store(pending);
  }
}

template <int MT, int KV>
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
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + meta);
  const uint32_t lut_bf = (uint32_t)__cvta_generic_to_shared(lut);
  const uint32_t zero_base = lut_bf + 1024;  // 512 zero bytes: activations of slots outside a pass
  uint8_t* xs = smem + meta + 1024 + 512;
  const size_t xs_bytes = (size_t)TR * pl.xs_stride * 2;
  const uint32_t xs_base = (uint32_t)__cvta_generic_to_shared(xs);
  const uint32_t red_base = xs_base + (uint32_t)((xs_bytes + 15) & ~(size_t)15);

  const uint32_t rank = cluster_rank();
  const int64_t cluster_id = blockIdx.x / pl.C;
  const int64_t nclusters = gridDim.x / pl.C;
  const int64_t r0 = (int64_t)blockIdx.y * TR;

  lut[threadIdx.x] = e4m3_to_bf16x2_bcast_x2p112(threadIdx.x);  // kThreads == 256 entries
  if (threadIdx.x < 128) lut[256 + threadIdx.x] = 0u;            // the zero block follows the table
  setup_slots(a, TR, r0, s_e, s_xr, s_pe, s_pm, &s_npass);
  // This CTA's K slice.
  const int cb = (int)((int64_t)pl.nchunk * rank / pl.C), ce = (int)((int64_t)pl.nchunk * (rank + 1) / pl.C);
  const bool use_bf16 = stage_x(a, pl, cb, ce, xs_base, s_e, s_xr);

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
    run_slabs<__nv_bfloat16, MT, KV>(a, pl, c, xs_base, red_base, lut_bf, zero_base, s_e, s_pm, r0, rank);
  else
    run_slabs<__half, MT, KV>(a, pl, c, xs_base, red_base, lut_bf, zero_base, s_e, s_pm, r0, rank);
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

constexpr size_t kSmemPerCta = 72 * 1024;  // three CTAs per SM
constexpr int kMaxCluster = 16;            // non-portable cluster sizes above 8

size_t smem_bytes(const Plan& p) {
  const size_t meta = ((size_t)p.TR * 24 + 15) & ~(size_t)15;
  const size_t xs = (((size_t)p.TR * p.xs_stride * 2) + 15) & ~(size_t)15;
  const size_t red = (size_t)2 * kSlabRows * p.TR * 4;
  return meta + 1024 + 512 + xs + red;
}

// Pick the K split C and the slabs per cluster. Time is modelled as (CTAs per
// SM) x (chunks per CTA + one chunk of per-slab synchronisation), with SMs
// holding fewer than two CTAs counted at half speed (too few warps to keep the
// memory system busy); slices must fit the shared-memory budget.
Plan choose_plan(Plan pl, int64_t row_tiles) {
  const int sms = sm_count();
  double best = 1e300;
  Plan out = pl;
  for (int C = 1; C <= kMaxCluster && C <= pl.nchunk; ++C) {
    const int per = (pl.nchunk + C - 1) / C;
    Plan p = pl;
    p.C = C;
    p.xs_stride = per * kChunkCols + 32;  // 512-byte multiple plus 64 bytes
    if (smem_bytes(p) > kSmemPerCta && C < kMaxCluster && C < pl.nchunk) continue;
    for (int64_t spc = 1; spc <= pl.slabs && spc <= 64; ++spc) {
      const int64_t nclusters = (pl.slabs + spc - 1) / spc;
      const int64_t ctas = nclusters * C * row_tiles;
      const double per_sm = (double)((ctas + sms - 1) / sms);
      const double eff = per_sm >= 2 ? 1.0 : 0.5;
      const double tm = per_sm * (double)spc * (per + 1) / eff;
      if (tm < best - 1e-9) {
        best = tm;
        out = p;
        out.spc = (int)spc;
      }
    }
  }
  return out;
}

template <int MT, int KV>
cudaError_t launch_kv(const QmvArgs& a, const Plan& pl, int64_t row_tiles, size_t smem, cudaStream_t st) {
  auto kern = qmv_cluster_kernel<MT, KV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (pl.C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const int64_t nclusters = (pl.slabs + pl.spc - 1) / pl.spc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nclusters * pl.C), (unsigned)row_tiles, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)pl.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, pl);
}

template <int MT>
cudaError_t launch_cluster(const QmvArgs& a, Plan pl, cudaStream_t st) {
  pl.TR = 8 * MT;
  const int64_t row_tiles = (a.R + pl.TR - 1) / pl.TR;
  pl = choose_plan(pl, row_tiles);
  const size_t smem = smem_bytes(pl);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;  // excluded by qmv_supported_k
  if (a.K % 64 == 0) return launch_kv<MT, 2>(a, pl, row_tiles, smem, st);
  if (a.K % 32 == 0) return launch_kv<MT, 1>(a, pl, row_tiles, smem, st);
  return launch_kv<MT, 0>(a, pl, row_tiles, smem, st);
}

}  // namespace

cudaError_t launch_qmv(const QmvArgs& a, int xdt, cudaStream_t st) {
  if (xdt == kF32) {
    const dim3 grid((unsigned)((a.N + kWarps - 1) / kWarps), (unsigned)((a.R + kF32Tokens - 1) / kF32Tokens));
    qmv_f32_kernel<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
  }
  if (qmv_stream_supported(a, xdt)) return launch_qmv_stream(a, xdt, st);
  if (qmv_group_supported(a, xdt)) return launch_qmv_group(a, xdt, st);
  if (qmv_tma_supported(a, xdt)) return launch_qmv_tma(a, xdt, st);
  Plan pl{};
  pl.nchunk = (int)((a.K + kChunkCols - 1) / kChunkCols);
  pl.slabs = (a.N + kSlabRows - 1) / kSlabRows;
  pl.x_is_bf16 = xdt == kBF16;
  // Rows per CTA tile: 8 for one- to eight-row calls and for gather calls,
  // 16 otherwise.
  const bool wide = a.rhs == nullptr && a.R > 8;
  if (wide) return launch_cluster<2>(a, pl, st);
  return launch_cluster<1>(a, pl, st);
}

// The staged slice (eight rows, K / 16 columns per CTA of a 16-CTA cluster)
// must fit one CTA's shared memory.
bool qmv_supported_k(int64_t K) { return K <= kQmvMaxK; }

}  // namespace nvfp4
