// Decode-shape NVFP4 products fed by TMA (K a multiple of 256).
//
// Same arithmetic, cluster K split and DSMEM reduction as the register-fed
// kernel in csrc/nvfp4_qmv.cu (QuantizedMatmul below the crossover and every
// GatherQMM decode; mlxcel PR #2629 "ROCm native NVFP4", Summary), but the
// packed weights and their E4M3 scales reach shared memory through TMA: one
// producer warp issues, per stage, a 2-D tile of 128 rows x 128 bytes of
// packed words (128-byte swizzle) and the matching 128 rows x 16 scale bytes.
// The bytes in flight are then set by the stage ring, not by registers, which
// is what a bandwidth-bound stream needs at HBM3e latency. Eight consumer
// warps read their m16n8k16 fragments from the ring (conflict-free thanks to
// the swizzle), decode and issue the MMAs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "nvfp4_qmv_common.cuh"

namespace nvfp4 {

__device__ int g_qmv_error = 0;  // first error code recorded by a bounded wait

namespace {
using namespace qmv;

constexpr int kConsumerWarps = kWarps;                     // 8 warps x 16 rows = one 128-row slab
constexpr int kTmaThreads = (kConsumerWarps + 1) * 32;     // plus one producer warp
constexpr int kMaxStages = 4;  // ring depth: the plan picks 2 to 4
constexpr uint32_t kWStage = kSlabRows * kChunkWords * 4;  // 16 KB of packed words
// Scale bytes arrive in blocks of eight chunks: one 128-byte-wide box of the
// scale plane per block (a 16-byte-wide box per chunk would cost the copy
// engine about as much as the chunk's 16 KB of words), 128-byte swizzled so
// the per-row 4-byte reads stay conflict-free; two blocks in flight.
constexpr int kScaleChunks = 8;
constexpr uint32_t kSBlock = kSlabRows * kScaleChunks * (kChunkCols / 16);  // 16 KB
constexpr int kSBlocks = 2;
// barriers: full[kMaxStages] empty[kMaxStages] sfull[kSBlocks] sempty[kSBlocks]
constexpr uint32_t kBarBytes = 8 * (2 * kMaxStages + 2 * kSBlocks);
constexpr uint64_t kWaitLimitNs = 2000000000ull;          // 2 s

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Consumer "stage empty" signal. Relaxed is enough: issue is in order and the
// arrive follows every instruction that consumed the stage's shared loads, so
// the reads have completed before the producer can see the arrival.
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// A waiting thread may be suspended by the hardware for up to this long per
// try (it resumes as soon as the phase completes), so waits do not burn issue
// slots that the working warps need.
constexpr uint32_t kSuspendHintNs = 1000;
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait; false once the limit passes (abort flag set, error recorded)
// or another warp has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int code) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(&g_qmv_error, 0, code);
        return false;
      }
    }
  }
}
// Bounded wait executed by all 32 lanes of a warp together: every lane polls
// the barrier (so each has acquired the phase), and the decision to stop is
// taken warp-wide, so the lanes never diverge on a timeout.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, int code, int* err) {
  if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t n = 1;; ++n) {
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
    if ((n & 63) == 0) {
      const bool stop = __any_sync(0xffffffffu, *abort_flag != 0 || gtimer() - t0 > kWaitLimitNs);
      if (stop) {
        if ((threadIdx.x & 31) == 0) {
          if (!*abort_flag) atomicCAS(err, 0, code);
          *abort_flag = 1;
        }
        return false;
      }
    }
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

struct TmaCtx {
  int64_t N;
  int64_t slab0, slab_step;
  int nslab, npass, cb, ce;
  const int* pass_e;
  const uint32_t* pass_m;
};

// Producer warp: walks the same job sequence as the consumers (slab, pass,
// chunk), lane 0 issuing the two TMA loads per stage; at every slab boundary
// the whole warp follows the consumers' cluster-barrier schedule.
__device__ void produce(const TmaCtx& c, const CUtensorMap* wmap, const CUtensorMap* smap, uint32_t wst,
                        uint32_t sst, uint32_t bars, volatile int* abort_flag, int kStages) {
  const int lane = threadIdx.x & 31;
  uint32_t u = 0;
  int s = 0;
  uint32_t ph = 0;
  uint32_t su = 0;  // scale blocks issued
  bool pending = false;
  const uint32_t sbars = bars + 8 * (2 * kMaxStages);
  for (int si = 0; si < c.nslab; ++si) {
    const int64_t slab = c.slab0 + (int64_t)si * c.slab_step;
    for (int p = 0; p < c.npass; ++p) {
      const int row = (int)((int64_t)c.pass_e[p] * c.N + slab * kSlabRows);
      for (int ch = c.cb; ch < c.ce; ++ch, ++u, s = (s + 1 == kStages ? 0 : s + 1), ph ^= (s == 0 ? 1u : 0u)) {
        if (lane == 0 && !*abort_flag) {
          if (((ch - c.cb) & (kScaleChunks - 1)) == 0) {  // scale block of chunks ch .. ch+7
            const uint32_t ss = su & 1u, sph = (su >> 1) & 1u;
            ++su;
            if (wait_bar(sbars + 8 * (kSBlocks + ss), sph ^ 1, abort_flag, 13)) {
              mbar_arrive_tx(sbars + 8 * ss, kSBlock);
              tma_load_2d(sst + ss * kSBlock, smap, ch * (kChunkCols / 16), row, sbars + 8 * ss);
            }
          }
          if (wait_bar(bars + 8 * (kStages + s), ph ^ 1, abort_flag, 11)) {  // stage empty
            mbar_arrive_tx(bars + 8 * s, kWStage);
            tma_load_2d(wst + (uint32_t)s * kWStage, wmap, ch * kChunkWords, row, bars + 8 * s);
          }
        }
      }
    }
    __syncwarp();
    if (pending) cluster_wait();
    cluster_arrive_relaxed();
    pending = true;
  }
  if (pending) cluster_wait();
  // No copy may still be in flight when the CTA leaves: wait (bounded) for
  // the last stages and scale blocks issued.
  if (lane == 0) {
    const uint32_t first = u > (uint32_t)kStages ? u - kStages : 0;
    for (uint32_t v = first; v < u; ++v) {
      const uint64_t t0 = gtimer();
      while (!mbar_try(bars + 8 * (v % kStages), (v / kStages) & 1) && gtimer() - t0 < kWaitLimitNs) {
      }
    }
    const uint32_t sfirst = su > (uint32_t)kSBlocks ? su - kSBlocks : 0;
    for (uint32_t v = sfirst; v < su; ++v) {
      const uint64_t t0 = gtimer();
      while (!mbar_try(sbars + 8 * (v & 1u), (v >> 1) & 1u) && gtimer() - t0 < kWaitLimitNs) {
      }
    }
  }
}

template <typename T, int MT>
__device__ void consume(const QmvArgs& a, const Plan& pl, const TmaCtx& c, uint32_t wst, uint32_t sst, uint32_t bars,
                        volatile int* abort_flag, uint32_t xs_base, uint32_t zero_base, uint32_t red_base,
                        uint32_t lut_bf, const int64_t* s_e, int64_t r0, uint32_t rank, const Corr* corr,
                        int ncorr) {
  const int kStages = pl.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int TR = pl.TR;
  const int rg = warp * 16 + g, rg8 = rg + 8;
  // swizzled offsets of this lane's two 16-byte chunks (2t, 2t+1) in rows rg, rg8
  const uint32_t oa0 = (uint32_t)rg * 128u + ((uint32_t)((2 * t) ^ (rg & 7)) << 4);
  const uint32_t oa1 = (uint32_t)rg * 128u + ((uint32_t)((2 * t + 1) ^ (rg & 7)) << 4);
  const uint32_t ob0 = (uint32_t)rg8 * 128u + ((uint32_t)((2 * t) ^ (rg8 & 7)) << 4);
  const uint32_t ob1 = (uint32_t)rg8 * 128u + ((uint32_t)((2 * t + 1) ^ (rg8 & 7)) << 4);
  // this lane's scale word in a scale block: row rg (rg8), 16-byte chunk
  // (chunk index within the block) ^ (row & 7), bytes 4t..4t+3
  const uint32_t osa = (uint32_t)rg * 128u + 4u * t, osb = (uint32_t)rg8 * 128u + 4u * t;

  constexpr int NA = NAcc<MT>::value;
  float acc[NA][MT][4];
#pragma unroll
  for (int k = 0; k < NA; ++k)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[k][mt][i] = 0.f;
  const uint32_t buf_bytes = (uint32_t)(kSlabRows * TR * 4);
  int buf = 0, pending = -1;
  int s = 0;        // ring stage of the next job
  uint32_t ph = 0;  // its phase parity
  uint32_t su = 0;  // scale blocks consumed
  const uint32_t sbars = bars + 8 * (2 * kMaxStages);

  ReduceOut red_out;
  auto gather = [&](uint32_t rb) { cluster_gather(pl.C, TR, rank, rb, threadIdx.x, kConsumerWarps * 32, red_out); };
  auto store = [&](int si) {
    cluster_store(a, pl.C, TR, pl.x_is_bf16, rank, c.slab0 + (int64_t)si * c.slab_step, s_e, r0, threadIdx.x,
                  kConsumerWarps * 32, red_out);
  };

  for (int si = 0; si < c.nslab; ++si) {
    for (int p = 0; p < c.npass; ++p) {
      const uint32_t pm = c.pass_m[p];
      uint32_t xa[MT], xstep[MT];
      int cur = 0;  // next residual correction (sorted by column)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int slot = g + 8 * mt;
        const bool in = slot < TR && ((pm >> slot) & 1);
        xa[mt] = in ? xs_base + 2u * (uint32_t)(slot * pl.xs_stride + 8 * t) : zero_base + 16u * (uint32_t)t;
        xstep[mt] = in ? 2u * kChunkCols : 0u;  // bytes per chunk (0: stay on the zero block)
      }
      for (int ch = c.cb; ch < c.ce; ++ch) {
        const int cs = s;          // this job's stage
        const uint32_t cph = ph;   // and its phase parity
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
        const int kb = (ch - c.cb) & (kScaleChunks - 1);  // chunk within its scale block
        const uint32_t sblk = su;                          // this chunk's scale block (running count)
        const uint32_t ss = sblk & 1u;
        const bool last_of_block = kb == kScaleChunks - 1 || ch + 1 == c.ce;
        if (last_of_block) ++su;
        uint32_t xc[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) xc[mt] = xa[mt] + xstep[mt] * (uint32_t)(ch - c.cb);
        if (kb == 0 && !wait_bar_warp(sbars + 8 * ss, (sblk >> 1) & 1u, abort_flag, 14, &g_qmv_error))
          continue;  // scale block full
        if (!wait_bar_warp(bars + 8 * cs, cph, abort_flag, 12, &g_qmv_error)) continue;  // stage full
        const uint32_t w = wst + (uint32_t)cs * kWStage, q = sst + ss * kSBlock;
        const uint32_t qa = q + osa + ((uint32_t)(kb ^ (rg & 7)) << 4), qb = q + osb + ((uint32_t)(kb ^ (rg8 & 7)) << 4);
        Chunk chk;
        chk.a0 = lds128(w + oa0);
        chk.a1 = lds128(w + oa1);
        chk.b0 = lds128(w + ob0);
        chk.b1 = lds128(w + ob1);
        chk.sa = lds32(qa);
        chk.sb = lds32(qb);
        compute_chunk<T, MT>(chk, xc, acc, lut_bf);
        // residuals of activations that f16 could not hold exactly
        const int cend = (ch - c.cb + 1) * kChunkCols;
        for (; cur < ncorr && corr[cur].col < cend; ++cur) {
          const Corr e = corr[cur];
          if (!((pm >> e.slot) & 1) || ((e.slot & 7) >> 1) != t) continue;
          const int kc = e.col - (ch - c.cb) * kChunkCols;
          const uint32_t wq = (uint32_t)(kc >> 5), wi = (uint32_t)((kc >> 3) & 3), sh = 4u * (uint32_t)(kc & 7);
          const uint32_t wa = lds32(w + (uint32_t)rg * 128u + ((wq ^ (uint32_t)(rg & 7)) << 4) + 4u * wi);
          const uint32_t wb = lds32(w + (uint32_t)rg8 * 128u + ((wq ^ (uint32_t)(rg8 & 7)) << 4) + 4u * wi);
          const uint32_t sa_w = lds32(qa - 4u * t + (uint32_t)(kc >> 4) / 4u * 4u);
          const uint32_t sb_w = lds32(qb - 4u * t + (uint32_t)(kc >> 4) / 4u * 4u);
          const uint32_t sbyte = 8u * ((uint32_t)(kc >> 4) & 3u);
          const float va = e2m1_to_f32((wa >> sh) & 0xF) * e4m3_to_f32((sa_w >> sbyte) & 0xFF);
          const float vb = e2m1_to_f32((wb >> sh) & 0xF) * e4m3_to_f32((sb_w >> sbyte) & 0xFF);
          const int lo = e.slot & 1;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if ((e.slot >> 3) != mt) continue;
            if (lo) {
              acc[0][mt][1] = fmaf(va, e.r, acc[0][mt][1]);
              acc[0][mt][3] = fmaf(vb, e.r, acc[0][mt][3]);
            } else {
              acc[0][mt][0] = fmaf(va, e.r, acc[0][mt][0]);
              acc[0][mt][2] = fmaf(vb, e.r, acc[0][mt][2]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_relaxed(bars + 8 * (kStages + cs));                   // stage empty
          if (last_of_block) mbar_arrive_relaxed(sbars + 8 * (kSBlocks + ss));  // scale block empty
        }
      }
    }
    // end of slab: reduce the previous slab over the cluster, publish this one
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
  }
  if (pending >= 0) {
    cluster_wait();
    gather(red_base + (uint32_t)(buf ^ 1) * buf_bytes);
    store(pending);
  }
}

// Dynamic shared memory: [1024-aligned] W stages | S stages | barriers (full[S],
// empty[S], abort) | meta | bf16 scale table | staged activations | partials.
size_t tma_smem_bytes(const Plan& p) {
  const size_t ring = (size_t)p.stages * kWStage + kSBlocks * kSBlock + kBarBytes + 16;
  const size_t meta = ((size_t)p.TR * 24 + 15) & ~(size_t)15;
  const size_t xs = (((size_t)p.xs_slots * p.xs_stride * 2) + 15) & ~(size_t)15;
  const size_t red = (size_t)2 * kSlabRows * p.TR * 4;
  return 1024 + ring + meta + 1024 + 512 + xs + red;
}

template <int MT>
__global__ void __launch_bounds__(kTmaThreads, 2)
qmv_tma_kernel(const QmvArgs a, const Plan pl, const __grid_constant__ CUtensorMap wmap,
               const __grid_constant__ CUtensorMap smap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  const int kStages = pl.stages;
  const uint32_t wst = base, sst = base + kStages * kWStage;  // both 1024-byte aligned (16 KB units)
  const uint32_t bars = sst + kSBlocks * kSBlock;
  const uint32_t ring_bytes = kStages * kWStage + kSBlocks * kSBlock;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bp + ring_bytes + kBarBytes);
  uint8_t* after = bp + ring_bytes + kBarBytes + 16;
  const int TR = pl.TR;
  int64_t* s_e = reinterpret_cast<int64_t*>(after);
  int64_t* s_xr = s_e + TR;
  int* s_pe = reinterpret_cast<int*>(s_xr + TR);
  uint32_t* s_pm = reinterpret_cast<uint32_t*>(s_pe + TR);
  __shared__ int s_npass;
  const size_t meta = ((size_t)TR * 24 + 15) & ~(size_t)15;
  uint32_t* lut = reinterpret_cast<uint32_t*>(after + meta);
  const uint32_t lut_bf = (uint32_t)__cvta_generic_to_shared(lut);
  const uint32_t zero_base = lut_bf + 1024;  // 512 zero bytes: activations of slots outside a pass
  const uint32_t xs_base = zero_base + 512;
  const size_t xs_bytes = (size_t)pl.xs_slots * pl.xs_stride * 2;
  const uint32_t red_base = xs_base + (uint32_t)((xs_bytes + 15) & ~(size_t)15);
  __shared__ Corr s_corr[kMaxCorr];
  __shared__ int s_ncorr;

  const uint32_t rank = cluster_rank();
  const int64_t cluster_id = blockIdx.x / pl.C;
  const int64_t nclusters = gridDim.x / pl.C;
  const int64_t r0 = (int64_t)blockIdx.y * TR;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars + 8 * s, 1);                            // full: producer arrive + TMA bytes
      mbar_init(bars + 8 * (kStages + s), kConsumerWarps);  // empty: one arrive per consumer warp
    }
    for (int b = 0; b < kSBlocks; ++b) {
      mbar_init(bars + 8 * (2 * kMaxStages + b), 1);
      mbar_init(bars + 8 * (2 * kMaxStages + kSBlocks + b), kConsumerWarps);
    }
    *abort_flag = 0;
    s_ncorr = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x == kConsumerWarps * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&smap)) : "memory");
  }
  if (threadIdx.x < 256) lut[threadIdx.x] = e4m3_to_bf16x2_bcast_x2p112(threadIdx.x);
  if (threadIdx.x < 128) lut[256 + threadIdx.x] = 0u;  // the zero block follows the table
  // Launched as a programmatic dependent (launch overlap on), this CTA may be
  // running while the previous kernel on the stream finishes. The next kernel
  // may start as soon as every CTA here has started; the weight planes are
  // read at once (the caller guarantees no running kernel writes them), the
  // gather indices and the activations only after the wait below (a no-op
  // without a programmatic dependency).
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.rhs != nullptr || a.lhs != nullptr) asm volatile("griddepcontrol.wait;" ::: "memory");
  setup_slots(a, TR, r0, s_e, s_xr, s_pe, s_pm, &s_npass);  // ends with __syncthreads

  const int cb = (int)((int64_t)pl.nchunk * rank / pl.C), ce = (int)((int64_t)pl.nchunk * (rank + 1) / pl.C);

  TmaCtx c;
  c.N = a.N;
  c.slab0 = cluster_id;
  c.slab_step = nclusters;
  c.nslab = (int)(cluster_id < pl.slabs ? (pl.slabs - cluster_id + nclusters - 1) / nclusters : 0);
  c.npass = s_npass;
  c.cb = cb;
  c.ce = ce;
  c.pass_e = s_pe;
  c.pass_m = s_pm;
  // The producer starts streaming weights at once; the consumer warps stage
  // the activations meanwhile (named barrier 1, 256 threads).
  if (warp == kConsumerWarps) {
    produce(c, &wmap, &smap, wst, sst, bars, abort_flag, kStages);
    cluster_arrive_relaxed();
    cluster_wait();
    return;
  }
  // column 64t+8q+i of a chunk is staged at chunk offset (4q+t)*8+i
  auto dst_of = [&](int slot, int ch, int w8) {
    return xs_base + 2u * (uint32_t)(slot * pl.xs_stride + ch * kChunkCols + (4 * (w8 & 7) + (w8 >> 3)) * 8);
  };
  asm volatile("griddepcontrol.wait;" ::: "memory");  // activations and outputs follow the previous kernel
  const int mode = stage_x_corr<0, kConsumerWarps * 32>(a, pl, cb, ce, dst_of, s_e, s_xr, s_corr, &s_ncorr);
  const bool use_bf16 = mode == 2;
  const int ncorr = mode == 1 ? s_ncorr : 0;
  if (use_bf16) {
    consume<__nv_bfloat16, MT>(a, pl, c, wst, sst, bars, abort_flag, xs_base, zero_base, red_base, lut_bf, s_e, r0,
                               rank, s_corr, 0);
  } else {
    consume<__half, MT>(a, pl, c, wst, sst, bars, abort_flag, xs_base, zero_base, red_base, lut_bf, s_e, r0, rank,
                        s_corr, ncorr);
  }
  // Peers may still read this CTA's partials: leave together.
  cluster_arrive();
  cluster_wait();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int sm_count() {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

// Launch plan: K split C (cluster size), slabs per cluster, ring depth.
// Modelled time (microseconds of one CTA's wall clock), its constants fitted
// to plan sweeps of the three decode shapes at 1, 4 and 16 tokens on GB300:
//   (waves + 0.3 (waves - 1)) * slabs_per_cluster * (chunks_per_slab * w(k) + sync(C, k))
// `capacity(C, smem)` is the number of CTAs that can be resident at once
// (clusters must fit a GPC, so a 7-CTA cluster packs worse than a 6-CTA
// one); k is the most CTAs an SM holds in a wave; w(1) = 0.4 and
// w(k) = 0.3 k per 16 KB chunk (CTAs on one SM share its copy engine and
// issue slots); a slab boundary costs a cluster barrier and the exchange of
// partial sums, 0.2 (1 + 0.1 C) k, doubled for sixteen token slots (0.2
// without peers). Sixteen token slots cost 1.6x per chunk, each further
// staged token 2% more.
template <typename CapFn>
Plan tma_plan(Plan pl, int64_t row_tiles, CapFn capacity) {
  const int sms = sm_count();
  double best = 1e300;
  Plan out = pl;
  out.C = 0;
  const double mt_factor = pl.TR > 8 ? 1.6 : 1.0 + 0.02 * (pl.xs_slots - 1);
  for (int C = 1; C <= 16 && C <= pl.nchunk; ++C)
    for (int stages = kMaxStages; stages >= 2; --stages) {
      const int per = (pl.nchunk + C - 1) / C;
      Plan p = pl;
      p.C = C;
      p.stages = stages;
      p.xs_stride = per * kChunkCols + 32;  // 512-byte multiple plus 64 bytes
      const int64_t cap = capacity(C, tma_smem_bytes(p));
      if (cap < 1) continue;
      const double depth = stages >= 4 ? 1.0 : stages == 3 ? 1.04 : 1.12;  // shallower rings hide less latency
      const double sync_c = C > 1 ? 0.2 * (1.0 + 0.1 * C) * (pl.TR > 8 ? 2.0 : 1.0) : 0.2;
      for (int64_t spc = 1; spc <= pl.slabs && spc <= 64; ++spc) {
        const int64_t ctas = (pl.slabs + spc - 1) / spc * C * row_tiles;
        const int64_t waves = (ctas + cap - 1) / cap;
        const int64_t wave_ctas = ctas < cap ? ctas : cap;
        const int64_t k = (wave_ctas + sms - 1) / sms;
        const double w = (k <= 1 ? 0.4 : 0.3 * (double)k) * depth * mt_factor;
        const double sync = C > 1 ? sync_c * (double)(k > 1 ? k : 1) : sync_c;
        const double tm = ((double)waves + 0.3 * (double)(waves - 1)) * (double)spc * ((double)per * w + sync);
        if (tm < best - 1e-9) {
          best = tm;
          out = p;
          out.spc = (int)spc;
        }
      }
    }
  return out;
}

template <int MT>
cudaError_t launch_mt(const QmvArgs& a, Plan pl, int64_t row_tiles, cudaStream_t st) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int64_t rows = a.E * a.N;
  CUtensorMap wmap, smap;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 8), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 2)};
    const cuuint32_t box[2] = {kChunkWords, kSlabRows};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(a.w), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 16), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 16)};
    const cuuint32_t box[2] = {kScaleChunks * (kChunkCols / 16), kSlabRows};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.scales), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kern = qmv_tma_kernel<MT>;
  int dev = 0;
  cudaGetDevice(&dev);
  // Plans are cached per device and shape: the first call on a shape sets the
  // kernel's shared-memory limit and asks the runtime how many CTAs of each
  // candidate size fit an SM (registers, shared memory and the per-block
  // reservation all count); later calls reuse the answer.
  using Key = std::tuple<int, int64_t, int64_t, int64_t, int64_t, int>;
  static std::mutex mu;
  static std::map<Key, Plan> cache;
  static std::map<int, int> max_dyn_of_dev;
  const Key key{dev, a.K, a.N, a.E, row_tiles * 64 + pl.xs_slots, pl.x_is_bf16};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      pl = it->second;
    } else {
      int max_dyn;
      auto md = max_dyn_of_dev.find(dev);
      if (md == max_dyn_of_dev.end()) {
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        max_dyn = optin - (int)fa.sharedSizeBytes;  // dynamic + static <= the opt-in limit
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
        if (e != cudaSuccess) return e;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
          return cudaGetLastError();
        max_dyn_of_dev[dev] = max_dyn;
      } else {
        max_dyn = md->second;
      }
      // CTAs of a C-CTA cluster launch that can be resident at once
      auto capacity = [&](int C, size_t smem) -> int64_t {
        if (smem > (size_t)max_dyn) return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(C * 64), 1, 1);
        cfg.blockDim = dim3(kTmaThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)C;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
          cudaGetLastError();
          return 0;
        }
        return (int64_t)n * C;
      };
      pl = tma_plan(pl, row_tiles, capacity);
      cache[key] = pl;
    }
  }
  if (pl.C == 0) return cudaErrorInvalidValue;
  const size_t smem = tma_smem_bytes(pl);
  const int64_t nclusters = (pl.slabs + pl.spc - 1) / pl.spc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nclusters * pl.C), (unsigned)row_tiles, 1);
  cfg.blockDim = dim3(kTmaThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)pl.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_overlap() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, a, pl, wmap, smap);
}

}  // namespace

bool qmv_tma_supported(const QmvArgs& a, int xdt) {
  // 16-bit activations; whole 256-column chunks (so the scale plane's row
  // pitch is a multiple of 16 bytes); 32-bit TMA row coordinates.
  return xdt != kF32 && a.K % 256 == 0 && a.K > 0 && a.E * a.N < (1ll << 31) && a.N > 0;
}

cudaError_t launch_qmv_tma(const QmvArgs& a, int xdt, cudaStream_t st) {
  Plan pl{};
  pl.nchunk = (int)(a.K / kChunkCols);
  pl.slabs = (a.N + kSlabRows - 1) / kSlabRows;
  pl.x_is_bf16 = xdt == kBF16;
  const bool wide = a.rhs == nullptr && a.R > 8;
  // Only the slots that exist get staging space (a one-row call stages one row).
  if (wide) {
    pl.TR = 16;
    pl.xs_slots = (int)(a.R < 16 ? a.R : 16);
    return launch_mt<2>(a, pl, (a.R + 15) / 16, st);
  }
  pl.TR = 8;
  pl.xs_slots = (int)(a.R < 8 ? a.R : 8);
  return launch_mt<1>(a, pl, (a.R + 7) / 8, st);
}

int read_qmv_error() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qmv_error, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  cudaMemcpyToSymbol(g_qmv_error, &zero, sizeof(int));
  return v;
}

}  // namespace nvfp4
