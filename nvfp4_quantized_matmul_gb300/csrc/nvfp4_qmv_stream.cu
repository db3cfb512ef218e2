// Decode-shape NVFP4 QuantizedMatmul as one persistent, evenly split weight
// stream: y = x @ dequantize(w).T * gs / 2688 for 1 to 16 token rows
// (mlxcel PR #2629 "ROCm native NVFP4", Summary: qmv for small M, the global
// scale applied once per output after the f32 sum).
//
// GB300 design.
//  * The product is bound by streaming the packed planes (9/16 byte per
//    weight). One CTA per SM, each with 16 consumer warps, one TMA producer
//    warp and one epilogue warp, holds a ring of 32 KB stages (256 weight rows
//    x 256 columns of packed words, 128-byte swizzled) plus 16 KB scale blocks
//    (256 rows x 4 chunks of E4M3 bytes, 64-byte swizzled): about 160 KB in
//    flight per SM, which is what HBM3e needs at its latency.
//  * Work split. The plane is a grid of tiles (256-row tile, 256-column
//    chunk). K is cut into S groups only as far as needed for the group's
//    activations to fit in shared memory (staged once per CTA, f16 when every
//    value converts exactly); each group's tiles, in row-major order, are
//    divided evenly over its CTAs (stream-K). A CTA therefore streams a
//    contiguous run of rows, every SM gets the same number of tiles to within
//    one, and no cluster or inter-CTA wait is involved.
//  * A row tile covered by one CTA is finished in place. A row tile split
//    between CTAs (by the even division or by the K groups) is finished by
//    whichever contributor arrives last: each adds its partial sums to the
//    tile's f32 workspace block with one bulk reduce-add of the copy engine,
//    then adds its chunk count to the tile's counter; the one that completes
//    the count (K / 256 chunks) reads the sums back, writes y and zeroes the
//    block and the counter for the next call. Nobody waits on another CTA.
//  * Math (shared with the other decode kernels): each weight word is decoded
//    exactly into f16 pairs that feed mma.sync m16n8k16 A fragments (weights
//    are the 16-row A operand, token rows the 8-wide B operand, f32
//    accumulation on the tensor pipe).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "nvfp4_pipe.cuh"
#include "nvfp4_qmv_common.cuh"

namespace nvfp4 {

__device__ int g_stream_error = 0;  // first error code recorded by a bounded wait

namespace {
using namespace qmv;
using namespace pipe;

constexpr int kTileRows = 256;               // weight rows per tile
// Warp roles for RT row tiles (16 rows each) per consumer warp: 16 / RT
// consumer warps, then the TMA producer warp, then the epilogue warp.
template <int RT> struct Geo {
  static constexpr int kCW = kTileRows / (16 * RT);
  static constexpr int kProducer = kCW;
  static constexpr int kEpilogue = kCW + 1;
  static constexpr int kThreads = (kCW + 2) * 32;
};
constexpr uint32_t kWBox = kTileRows * 128;  // one chunk of words: 256 rows x 128 B
constexpr int kSChunks = 4;                  // chunks per scale block
constexpr uint32_t kSBox = kTileRows * 64;   // one scale block: 256 rows x 64 B
constexpr int kMaxStages = 6;
constexpr int kAccSlots = 16;  // workspace floats per weight row (token slots)
// A partial-sum buffer holds, per token slot, the 256 row sums of a tile
// (1 KB); the slots follow one another, so a tile's sums for M token rows are
// M KB contiguous, as in the workspace (tile-major: tile r's block is
// [16 slots][256 rows] floats at r * 16 KB), and move with one bulk copy.
constexpr uint32_t kPStride = kTileRows;
// barriers: full[kMaxStages] empty[kMaxStages] sfull[2] sempty[2] pfull[2]
// pempty[2] back[1], rounded to 16 bytes (what follows is read 16 B at a time)
constexpr uint32_t kBarBytes = ((2 * kMaxStages + 9) * 8 + 15) / 16 * 16;

// Launch plan (host).
struct SPlan {
  int M;          // token rows, 1..16
  int nc;         // 256-column chunks in K
  int ncg;        // chunks per K group
  int S;          // K groups
  int gs;         // CTAs per group
  int64_t nrt;    // 256-row tiles
  int stages;     // word stages in the ring
  int xs_chunks;  // most chunks of activations a CTA stages
  int xs_stride;  // staged activation row stride, elements (= 32 mod 256)
  int x_is_bf16;  // activation (and output) dtype is bf16, else f16
  int pslots;     // token slots held in a partial-sum buffer (8 per MMA tile)
  // Fused gate/up (GLU) launches: the plane holds 2 * glu_cols rows (gate
  // rows, then up rows); row tile r stands for gate rows [128 r, 128 r + 128)
  // stacked on the matching up rows, and writes act(gate) * up for those
  // glu_cols-wide output columns. glu_act: 1 SiLU, 2 GELU (tanh form).
  int64_t glu_cols;
  int glu_act;
  // Limit of every bounded wait of the launch (2 s unless a test shortens
  // it), and, for tests of that limit only, a flag that makes consumer warp 0
  // of CTA 0 withhold its release of its first stage, so that the producer's
  // wait for that stage runs out.
  uint64_t wait_ns;
  int withhold;
};

struct Seg {
  int64_t r;  // row tile
  int c0, c1;  // chunks [c0, c1) of the CTA's K group
};
// A CTA's work within its K group, as tile ranges in row-major tile order
// (tile = row tile * ncg + chunk). The group's row tiles are dealt out whole,
// W = nrt / gs consecutive ones per CTA; the nrt mod gs left over are split
// evenly over all the group's CTAs by tiles. Each CTA does its share of the
// split rows first, so that finishing those (shared with other CTAs) overlaps
// the streaming of its whole rows, which it completes alone.
struct Work {
  int64_t a0, a1;  // share of the split rows
  int64_t b0, b1;  // whole rows
  int ncg;
  __device__ __forceinline__ static Work of(const SPlan& p, int gi) {
    Work w;
    const int64_t W = p.nrt / p.gs, whole = W * p.gs * p.ncg, rest = (p.nrt - W * p.gs) * p.ncg;
    w.a0 = whole + rest * gi / p.gs;
    w.a1 = whole + rest * (gi + 1) / p.gs;
    w.b0 = (int64_t)gi * W * p.ncg;
    w.b1 = w.b0 + W * p.ncg;
    w.ncg = p.ncg;
    return w;
  }
  __device__ __forceinline__ bool next(Seg& s) {
    const bool first = a0 < a1;
    if (!first && b0 >= b1) return false;
    const int64_t t = first ? a0 : b0, t1 = first ? a1 : b1;
    s.r = t / ncg;
    s.c0 = (int)(t % ncg);
    const int64_t left = t1 - t;
    s.c1 = left < (int64_t)(ncg - s.c0) ? s.c0 + (int)left : ncg;
    if (first)
      a0 = t + (s.c1 - s.c0);
    else
      b0 = t + (s.c1 - s.c0);
    return true;
  }
};

struct Bars {
  uint32_t base;
  int ns;
  __device__ __forceinline__ uint32_t full(uint32_t s) const { return base + 8u * s; }
  __device__ __forceinline__ uint32_t empty(uint32_t s) const { return base + 8u * (kMaxStages + s); }
  __device__ __forceinline__ uint32_t sfull(uint32_t b) const { return base + 8u * (2 * kMaxStages + b); }
  __device__ __forceinline__ uint32_t sempty(uint32_t b) const { return base + 8u * (2 * kMaxStages + 2 + b); }
  __device__ __forceinline__ uint32_t pfull(uint32_t b) const { return base + 8u * (2 * kMaxStages + 4 + b); }
  __device__ __forceinline__ uint32_t pempty(uint32_t b) const { return base + 8u * (2 * kMaxStages + 6 + b); }
  __device__ __forceinline__ uint32_t back() const { return base + 8u * (2 * kMaxStages + 8); }
};

// The chunks of its K group a CTA visits form a circular run: staged chunk j
// holds group chunk (first + j) mod ncg, j < count. Whole rows visit them all.
struct XRun {
  int first, count;
};
__device__ __forceinline__ XRun x_run(const SPlan& p, const Work& wk) {
  if (wk.b1 > wk.b0 || wk.a1 - wk.a0 >= p.ncg) return XRun{0, p.ncg};
  return XRun{(int)(wk.a0 % p.ncg), (int)(wk.a1 - wk.a0)};
}

// Stages the CTA's run of activation columns for every token row, 8 columns
// per 16-byte unit, column 64t+8q+i of a chunk at chunk offset (4q+t)*8+i.
// bf16 inputs are staged as f16 when that is exact; a value f16 cannot hold
// exactly but within its range is split into its f16 part and an f32
// residual (up to kMaxCorr of them, recorded by group-relative column and
// sorted); otherwise the bf16 values are staged. Returns 0 (f16), 1 (f16 with
// residuals) or 2 (bf16). Threads 0 .. kN-1 (the consumer warps) take part;
// *n_corr must be zero and visible on entry. Loads are issued four at a time
// per thread so that their latencies overlap. Token slot s reads activation
// row s, or xrow[s] for an expert group (kGrp). kCoherent loads through L2
// only (activations written earlier in the same launch).
template <int kN, bool kGrp, bool kCoherent = false>
__device__ int stage_run(const QmvArgs& a, const SPlan& p, int chunk0, XRun run, uint32_t xs_base, Corr* corr,
                         int* n_corr, const int64_t* xrow) {
  constexpr int kBatch = 4;
  const int per_slot = run.count * (kChunkCols / 8), units = p.M * per_slot;
  const int tid = (int)threadIdx.x;
  const uint16_t* xg = static_cast<const uint16_t*>(a.x);
  auto locate = [&](int u, int64_t& src, uint32_t& dst, int& gcol) {
    const int slot = u / per_slot, rem = u % per_slot, j = rem >> 5, w8 = rem & 31;
    int gc = run.first + j;
    if (gc >= p.ncg) gc -= p.ncg;
    gcol = gc * kChunkCols + 8 * w8;  // group-relative column
    src = (kGrp ? xrow[slot] : (int64_t)slot) * a.K + (int64_t)chunk0 * kChunkCols + gcol;
    dst = xs_base + 2u * (uint32_t)(slot * p.xs_stride + j * kChunkCols + (4 * (w8 & 7) + (w8 >> 3)) * 8);
  };
  int hard = 0;
  for (int u0 = tid; u0 < units; u0 += kBatch * kN) {
    uint4 v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int u = u0 + b * kN;
      v[b] = make_uint4(0, 0, 0, 0);
      if (u < units) {
        int64_t src;
        uint32_t dst;
        int gcol;
        locate(u, src, dst, gcol);
        v[b] = kCoherent ? __ldcg(reinterpret_cast<const uint4*>(xg + src))
                         : __ldg(reinterpret_cast<const uint4*>(xg + src));
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int u = u0 + b * kN;
      if (u >= units) continue;
      int64_t src;
      uint32_t dst;
      int gcol;
      locate(u, src, dst, gcol);
      uint4 o = v[b];
      if (p.x_is_bf16) {
        const uint32_t in[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
        uint32_t h2[4];
        // Fast path, integer only: a bf16 whose exponent field e lies in
        // f16's normal range (113 <= e <= 142) is exactly the f16 with
        // exponent e - 112 and the same seven fraction bits (padded with
        // zeros), i.e. its magnitude bits minus 112 << 7, shifted left by 3.
        // The range test adds 0x8000 - 0x3880 to each 15-bit magnitude (the
        // 0x8000 keeps a borrow from crossing halves): inside the range the
        // result is 0x8000..0x8EFF. Any other value (zero, f16 subnormal or
        // beyond f16, NaN) takes the exact float path below.
        bool fast = true;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t m = in[q] & 0x7FFF7FFFu;
          const uint32_t d = (m | 0x80008000u) - 0x38803880u;
          fast &= (d & 0xF000F000u) == 0x80008000u && (((d & 0x0F000F00u) + 0x01000100u) & 0x10001000u) == 0u;
          h2[q] = (in[q] & 0x80008000u) | ((m - 0x38003800u) << 3);
        }
        if (!fast) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = __uint_as_float(in[q] << 16), hi = __uint_as_float(in[q] & 0xFFFF0000u);
            const __half2 h = __floats2half2_rn(lo, hi);
            const float2 back = __half22float2(h);
            h2[q] = *reinterpret_cast<const uint32_t*>(&h);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float xv = e ? hi : lo, bv = e ? back.y : back.x;
              if (bv != xv) {
                if (!(fabsf(xv) <= 65504.f)) {  // beyond f16's range, or NaN
                  hard = 1;
                } else {
                  const int i = atomicAdd(n_corr, 1);
                  if (i < kMaxCorr)
                    corr[i] = Corr{u / per_slot, gcol + 2 * q + e, xv - bv};
                  else
                    hard = 1;
                }
              }
            }
          }
        }
        o = make_uint4(h2[0], h2[1], h2[2], h2[3]);
      }
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w));
    }
  }
  if (sync_or<kN>(hard)) {  // keep the exact bf16 activations instead
    for (int u0 = tid; u0 < units; u0 += kBatch * kN) {
      uint4 v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int u = u0 + b * kN;
        v[b] = make_uint4(0, 0, 0, 0);
        if (u < units) {
          int64_t src;
          uint32_t dst;
          int gcol;
          locate(u, src, dst, gcol);
          v[b] = kCoherent ? __ldcg(reinterpret_cast<const uint4*>(xg + src))
                           : __ldg(reinterpret_cast<const uint4*>(xg + src));
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int u = u0 + b * kN;
        if (u >= units) continue;
        int64_t src;
        uint32_t dst;
        int gcol;
        locate(u, src, dst, gcol);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v[b].x), "r"(v[b].y), "r"(v[b].z),
                     "r"(v[b].w));
      }
    }
    sync_all<kN>();
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
  sync_all<kN>();
  return 1;
}

// Position in a CTA's chunk sequence (the order every role walks).
struct ChunkPos {
  Work wk;
  Seg sg;
  int c;
  bool valid;
  __device__ __forceinline__ void start(const Work& w) {
    wk = w;
    valid = wk.next(sg);
    c = valid ? sg.c0 : 0;
  }
  __device__ __forceinline__ void advance() {
    if (valid && ++c >= sg.c1) {
      valid = wk.next(sg);
      if (valid) c = sg.c0;
    }
  }
  // the scale block covering this chunk is loaded here (segment start or a
  // block boundary)
  __device__ __forceinline__ bool block_start(int ac) const { return c == sg.c0 || ac % kSChunks == 0; }
};

// Ring positions of the producer (copies issued, next word stage and its
// phase, scale blocks issued). A launch that runs several calls keeps one
// across them: the ring never drains between calls.
struct ProdState {
  uint32_t u = 0, s = 0, ph = 0, su = 0;
};

// Producer (lane 0 of the producer warp): the same chunk walk as the
// consumers; a scale block at the start of each segment and at every fourth
// chunk, a word stage per chunk. An expert group (kGrp) reads its expert's
// plane through 3-D maps ([E, N, K] planes, rows past N zero-filled).
// Returns false once a wait gave up.
template <bool kGrp, bool kGlu>
__device__ bool produce(const SPlan& p, int grp, Work wk, const CUtensorMap* wmap,
                        const CUtensorMap* smap, uint32_t wst, uint32_t sst, const Bars& bar,
                        volatile int* abort_flag, int expert, ProdState& st, int stages) {
  uint32_t &u = st.u, &s = st.s, &ph = st.ph, &su = st.su;
  ChunkPos pos;
  pos.start(wk);
  for (; pos.valid; pos.advance()) {
    const int ac = grp * p.ncg + pos.c;  // absolute chunk
    // GLU: the tile's gate half-tile; its up half-tile is glu_cols rows on
    const int row = (int)(pos.sg.r * (kGlu ? kTileRows / 2 : kTileRows));
    const int up_row = (int)(p.glu_cols + row);
    if (pos.block_start(ac)) {
      const uint32_t b = su & 1u, bph = (su >> 1) & 1u;
      if (!wait_bar(bar.sempty(b), bph ^ 1u, abort_flag, 21, &g_stream_error, p.wait_ns)) return false;
      ++su;
      mbar_arrive_tx(bar.sfull(b), kSBox);
      if (kGlu) {
        tma_load_2d(sst + b * kSBox, smap, (ac / kSChunks) * (kSChunks * 16), row, bar.sfull(b));
        tma_load_2d(sst + b * kSBox + kSBox / 2, smap, (ac / kSChunks) * (kSChunks * 16), up_row, bar.sfull(b));
      } else if (kGrp)
        tma_load_3d(sst + b * kSBox, smap, (ac / kSChunks) * (kSChunks * 16), row, expert, bar.sfull(b));
      else
        tma_load_2d(sst + b * kSBox, smap, (ac / kSChunks) * (kSChunks * 16), row, bar.sfull(b));
    }
    if (!wait_bar(bar.empty(s), ph ^ 1u, abort_flag, 22, &g_stream_error, p.wait_ns)) return false;
    ++u;
    mbar_arrive_tx(bar.full(s), kWBox);
    if (kGlu) {
      tma_load_2d(wst + s * kWBox, wmap, ac * kChunkWords, row, bar.full(s));
      tma_load_2d(wst + s * kWBox + kWBox / 2, wmap, ac * kChunkWords, up_row, bar.full(s));
    } else if (kGrp)
      tma_load_3d(wst + s * kWBox, wmap, ac * kChunkWords, row, expert, bar.full(s));
    else
      tma_load_2d(wst + s * kWBox, wmap, ac * kChunkWords, row, bar.full(s));
    if (++s == (uint32_t)stages) {
      s = 0;
      ph ^= 1u;
    }
  }
  return true;
}

// No copy may still be in flight when the CTA exits: waits (bounded) for the
// last ring's worth of copies the producer issued.
__device__ __forceinline__ void drain_copies(const ProdState& st, const Bars& bar, int stages) {
  const uint32_t first = st.u > (uint32_t)stages ? st.u - stages : 0;
  for (uint32_t v = first; v < st.u; ++v) wait_bar_quiet(bar.full(v % stages), (v / stages) & 1u);
  const uint32_t sfirst = st.su > 2u ? st.su - 2u : 0;
  for (uint32_t v = sfirst; v < st.su; ++v) wait_bar_quiet(bar.sfull(v & 1u), (v >> 1) & 1u);
}

// Accumulator sets per (row tile, token tile): consecutive k-steps rotate over
// them so that the MMAs form several dependency chains; two row tiles per warp
// already give two chains each.
template <int MT, int RT> struct NAccS {
  static constexpr int value = RT == 1 ? NAcc<MT>::value : (MT == 1 ? 2 : 1);
};

// One chunk for RT row tiles of 16 rows: the activation fragments of each
// half-chunk are loaded once and feed the MMAs of every row tile (same lane
// layout as compute_chunk: lane t's word j holds columns 64t+8j..+7, k-step s
// uses columns 64t+4s+0..3).
template <typename T, int MT, int RT, int NA>
__device__ __forceinline__ void compute_rt(const Chunk (&ch)[RT], const uint32_t (&xaddr)[MT],
                                           float (&acc)[NA][RT][MT][4], uint32_t lut_bf) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint4 xv[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[mt][q] = lds128(xaddr[mt] + 64 * (4 * half + q));
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const uint4& wa = half ? ch[rt].a1 : ch[rt].a0;
      const uint4& wb = half ? ch[rt].b1 : ch[rt].b0;
      uint32_t sa0, sa1, sb0, sb1;
      scale_pair<T>(ch[rt].sa, half, lut_bf, sa0, sa1);
      scale_pair<T>(ch[rt].sb, half, lut_bf, sb0, sb1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t da[4], db[4];
        Dt<T>::decode(u4get(wa, j), j < 2 ? sa0 : sa1, da);
        Dt<T>::decode(u4get(wb, j), j < 2 ? sb0 : sb1, db);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int sl = 2 * j + h;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t b0 = u4get(xv[mt][sl >> 1], 2 * (sl & 1));
            const uint32_t b1 = u4get(xv[mt][sl >> 1], 2 * (sl & 1) + 1);
            MmaOp<T>::run(acc[(8 * half + sl) % NA][rt][mt], da[2 * h], db[2 * h], da[2 * h + 1], db[2 * h + 1], b0,
                          b1);
          }
        }
      }
    }
  }
}

// Ring positions of a consumer warp (word stage and its phase, scale
// blocks, partial buffers handed over), kept across the calls of a launch.
struct ConsState {
  uint32_t s = 0, ph = 0, su = 0, pc = 0;
};

// Consumer warp: RT row tiles of 16 rows (rows 16 RT w .. 16 RT w + 16 RT - 1
// of the 256-row tile) over every chunk of the CTA's walk.
template <typename T, int MT, int RT>
__device__ void consume(const SPlan& p, int grp, Work wk, XRun run, uint32_t wst, uint32_t sst,
                        uint32_t pbuf, uint32_t pbuf_bytes, const Bars& bar, volatile int* abort_flag,
                        uint32_t xs_base, uint32_t zero_base, uint32_t lut_bf, const Corr* corr, int ncorr,
                        ConsState& cst, int stages) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  // 128-byte swizzle of the word stage: 16-byte granule j of row r sits at
  // j ^ (r & 7); this lane reads granules 2t and 2t+1 of rows rg and rg + 8.
  // 64-byte swizzle of a scale block: granule kb (chunk kb of the block) of
  // row r sits at kb ^ ((r >> 1) & 3); this lane reads its word t (groups
  // 4t..4t+3 of the chunk).
  int rg[RT];
  uint32_t oa0[RT], oa1[RT], ob0[RT], ob1[RT], osa[RT], osb[RT], swa[RT], swb[RT];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    rg[rt] = warp * 16 * RT + 16 * rt + g;
    const int ra = rg[rt], rb = ra + 8;
    oa0[rt] = (uint32_t)ra * 128u + ((uint32_t)((2 * t) ^ (ra & 7)) << 4);
    oa1[rt] = (uint32_t)ra * 128u + ((uint32_t)((2 * t + 1) ^ (ra & 7)) << 4);
    ob0[rt] = (uint32_t)rb * 128u + ((uint32_t)((2 * t) ^ (rb & 7)) << 4);
    ob1[rt] = (uint32_t)rb * 128u + ((uint32_t)((2 * t + 1) ^ (rb & 7)) << 4);
    osa[rt] = (uint32_t)ra * 64u + 4u * t;
    osb[rt] = (uint32_t)rb * 64u + 4u * t;
    swa[rt] = (uint32_t)((ra >> 1) & 3);
    swb[rt] = (uint32_t)((rb >> 1) & 3);
  }

  uint32_t xa[MT], xstep[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int slot = g + 8 * mt;
    const bool in = slot < p.M;
    xa[mt] = in ? xs_base + 2u * (uint32_t)(slot * p.xs_stride + 8 * t) : zero_base + 16u * (uint32_t)t;
    xstep[mt] = in ? 2u * kChunkCols : 0u;
  }

  constexpr int NA = NAccS<MT, RT>::value;
  float acc[NA][RT][MT][4];
  uint32_t &s = cst.s, &ph = cst.ph, &su = cst.su, &pc = cst.pc;
  bool hold = p.withhold && blockIdx.x == 0 && warp == 0;  // tests of the bounded waits only
  Seg sg;
  while (wk.next(sg)) {
#pragma unroll
    for (int k = 0; k < NA; ++k)
#pragma unroll
      for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[k][rt][mt][i] = 0.f;
    int cur = 0;  // next residual correction (sorted by column)
    while (cur < ncorr && corr[cur].col < sg.c0 * kChunkCols) ++cur;
    for (int c = sg.c0; c < sg.c1; ++c) {
      const int ac = grp * p.ncg + c, kb = ac % kSChunks;
      const uint32_t cs = s, cph = ph;  // this chunk's stage
      if (++s == (uint32_t)stages) {
        s = 0;
        ph ^= 1u;
      }
      const uint32_t sb = su & 1u, sph = (su >> 1) & 1u;
      const bool first_of_block = c == sg.c0 || kb == 0;
      const bool last_of_block = c + 1 == sg.c1 || kb == kSChunks - 1;
      if (last_of_block) ++su;
      if (first_of_block && !wait_bar_warp(bar.sfull(sb), sph, abort_flag, 23, &g_stream_error, p.wait_ns)) continue;
      if (!wait_bar_warp(bar.full(cs), cph, abort_flag, 24, &g_stream_error, p.wait_ns)) continue;
      const uint32_t w = wst + cs * kWBox, q = sst + sb * kSBox;
      Chunk chk[RT];
      uint32_t qa[RT], qb[RT];
#pragma unroll
      for (int rt = 0; rt < RT; ++rt) {
        qa[rt] = q + osa[rt] + (((uint32_t)kb ^ swa[rt]) << 4);
        qb[rt] = q + osb[rt] + (((uint32_t)kb ^ swb[rt]) << 4);
        chk[rt].a0 = lds128(w + oa0[rt]);
        chk[rt].a1 = lds128(w + oa1[rt]);
        chk[rt].b0 = lds128(w + ob0[rt]);
        chk[rt].b1 = lds128(w + ob1[rt]);
        chk[rt].sa = lds32(qa[rt]);
        chk[rt].sb = lds32(qb[rt]);
      }
      uint32_t xc[MT];
      const int jx = c >= run.first ? c - run.first : c - run.first + p.ncg;  // staged chunk
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) xc[mt] = xa[mt] + xstep[mt] * (uint32_t)jx;
      compute_rt<T, MT, RT, NA>(chk, xc, acc, lut_bf);
      // residuals of activations that f16 could not hold exactly
      const int cend = (c + 1) * kChunkCols;
      for (; cur < ncorr && corr[cur].col < cend; ++cur) {
        const Corr e = corr[cur];
        if (((e.slot & 7) >> 1) != t) continue;
        const int kc = e.col - c * kChunkCols;  // column within the chunk
        const uint32_t wq = (uint32_t)(kc >> 5), wi = (uint32_t)((kc >> 3) & 3), sh = 4u * (uint32_t)(kc & 7);
        const uint32_t grpb = (uint32_t)(kc >> 4);  // 16-column group within the chunk: byte of the granule
        const uint32_t sbyte = 8u * (grpb & 3u);
        const bool odd = e.slot & 1;
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
          const int ra = rg[rt], rb = ra + 8;
          const uint32_t wa = lds32(w + (uint32_t)ra * 128u + ((wq ^ (uint32_t)(ra & 7)) << 4) + 4u * wi);
          const uint32_t wb = lds32(w + (uint32_t)rb * 128u + ((wq ^ (uint32_t)(rb & 7)) << 4) + 4u * wi);
          const uint32_t sa_w = lds32(qa[rt] - 4u * t + 4u * (grpb >> 2));
          const uint32_t sb_w = lds32(qb[rt] - 4u * t + 4u * (grpb >> 2));
          // fp4 * e4m3 * residual is exact in f32 (at most 6 + 8 significant bits)
          const float da = e2m1_to_f32((wa >> sh) & 0xF) * e4m3_to_f32((sa_w >> sbyte) & 0xFF) * e.r;
          const float db = e2m1_to_f32((wb >> sh) & 0xF) * e4m3_to_f32((sb_w >> sbyte) & 0xFF) * e.r;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {  // selects, not indexing: the accumulators stay in registers
            const bool on = (e.slot >> 3) == mt;
            acc[0][rt][mt][0] += on && !odd ? da : 0.f;
            acc[0][rt][mt][1] += on && odd ? da : 0.f;
            acc[0][rt][mt][2] += on && !odd ? db : 0.f;
            acc[0][rt][mt][3] += on && odd ? db : 0.f;
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (!hold) mbar_arrive_relaxed(bar.empty(cs));
        if (last_of_block) mbar_arrive_relaxed(bar.sempty(sb));
      }
      hold = false;
    }
    // hand the segment's sums to the epilogue warp
    const uint32_t b = pc & 1u, bph = (pc >> 1) & 1u;
    ++pc;
    if (!wait_bar_warp(bar.pempty(b), bph ^ 1u, abort_flag, 25, &g_stream_error, p.wait_ns)) continue;
    const uint32_t pb = pbuf + b * pbuf_bytes;
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = rg[rt] + ((i & 2) ? 8 : 0);
          const int slot = 8 * mt + 2 * t + (i & 1);
          float v = 0.f;
#pragma unroll
          for (int k = 0; k < NA; ++k) v += acc[k][rt][mt][i];
          sts_f32(pb + 4u * ((uint32_t)slot * kPStride + (uint32_t)row), v);
        }
    mbar_arrive(bar.pfull(b));  // every lane: releases its own stores
  }
}

__device__ __forceinline__ void store_out(void* y, int is_bf16, int64_t idx, float v) {
  if (is_bf16)
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
  else
    static_cast<__half*>(y)[idx] = __float2half_rn(v);
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Element-wise float add of `bytes` of shared memory into global memory,
// performed by the copy engine at L2 (the split-tile reduction).
__device__ __forceinline__ void bulk_add_s2g(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Eight consecutive outputs (idx a multiple of 8, so 16-byte aligned).
__device__ __forceinline__ void store_out8(void* y, int is_bf16, int64_t idx, const float (&v)[8]) {
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (is_bf16) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
      o[q] = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const __half2 h = __floats2half2_rn(v[2 * q], v[2 * q + 1]);
      o[q] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + idx) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Epilogue warp: finishes each segment the consumers hand over. The
// workspace is tile-major: a split row tile owns a block of 16 slots x 256
// rows of float sums, of which a call with M token rows uses the first M KB.
// A dense call's row tile r uses block r. An expert group (kGrp) uses blocks
// wsbase .. wsbase + gs - 1, one per row tile left over after the whole rows
// are dealt out (there are fewer than gs), and writes token slot s to output
// row yrow[s] with the expert's global scale. A GLU tile (kGlu) holds gate
// sums in rows 0..127 and the matching up sums in rows 128..255 and writes
// act(factor * gate) * (factor * up) to output columns 128 r .. 128 r + 127.
// SiLU: v * sigmoid(v). GELU, tanh form: 0.5 v (1 + tanh(a)) with a =
// sqrt(2/pi) (v + 0.044715 v^3), written as v * sigmoid(2 a) (the same value:
// 0.5 (1 + tanh(a)) = 1 / (1 + exp(-2 a))). The fast exponential and divide
// keep the single epilogue warp's per-output cost low; their error (a few
// f32 ulp) is far below the output's 16-bit rounding.
__device__ __forceinline__ float glu_act(int act, float v) {
  const float z = act == 1 ? v : 1.5957691216057308f * (v + 0.044715f * v * v * v);
  return __fdividef(v, 1.0f + __expf(-z));
}

// Positions of the epilogue warp (partial buffers taken, read-backs), kept
// across the calls of a launch.
struct FinState {
  uint32_t pc = 0, bc = 0;
};

template <bool kGrp, bool kGlu>
__device__ void finish(const QmvArgs& a, const SPlan& p, Work wk, uint32_t pbuf, uint32_t pbuf_bytes,
                       const Bars& bar, volatile int* abort_flag, float* __restrict__ acc,
                       uint32_t* __restrict__ cnt, int expert, int wsbase, const int64_t* yrow, FinState& fst) {
  const int lane = threadIdx.x & 31;
  const float factor = global_factor(a.gs, kGrp ? expert : 0);
  const int64_t first_split = (p.nrt / p.gs) * p.gs;  // row tiles from here on may be split
  const bool has_gs = a.gs != nullptr;
  const int M = p.M;
  constexpr uint32_t kSlotBytes = kTileRows * 4u;
  const uint32_t tile_bytes = (uint32_t)M * kSlotBytes;  // this call's part of a tile block
  uint32_t &pc = fst.pc, &bc = fst.bc;
  Seg sg;
  while (wk.next(sg)) {
    const uint32_t b = pc & 1u, bph = (pc >> 1) & 1u;
    ++pc;
    if (!wait_bar_warp(bar.pfull(b), bph, abort_flag, 26, &g_stream_error, p.wait_ns)) break;
    const uint32_t pb = pbuf + b * pbuf_bytes;
    const int64_t n0 = sg.r * (kGlu ? kTileRows / 2 : kTileRows);
    const int64_t ncols = kGlu ? p.glu_cols : a.N;  // output columns
    const int rows = kGlu ? (int)(ncols - n0 < kTileRows / 2 ? ncols - n0 : kTileRows / 2)
                          : (int)(a.N - n0 < kTileRows ? a.N - n0 : kTileRows);
    bool own = p.S == 1 && sg.c0 == 0 && sg.c1 == p.ncg;  // the whole row tile is this CTA's
    const int64_t wt = kGrp ? wsbase + (sg.r - first_split) : sg.r;  // the tile's workspace block
    float* blk = acc + wt * (int64_t)(kAccSlots * kTileRows);
    if (!own) {
      // Add this piece to the tile's workspace sums with one bulk add (rows
      // past N add zeros), then count its chunks in.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // consumers' stores -> copy engine
      if (lane == 0) {
        bulk_add_s2g(blk, pb, tile_bytes);
        bulk_commit();
        bulk_wait_all();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        const uint32_t add = (uint32_t)(sg.c1 - sg.c0);
        own = atomicAdd(cnt + wt, add) + add == (uint32_t)p.nc;  // the last contribution finishes the tile
      }
      own = __shfl_sync(0xffffffffu, (int)own, 0) != 0;
      if (own) {
        // Bring the completed sums into this buffer, clear the workspace rows
        // and the counter for the next call.
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        if (lane == 0) {
          mbar_arrive_tx(bar.back(), tile_bytes);
          bulk_g2s(pb, blk, tile_bytes, bar.back());
        }
        const bool ok = wait_bar_warp(bar.back(), bc & 1u, abort_flag, 27, &g_stream_error, p.wait_ns);
        ++bc;
        if (!ok) {
          wait_bar_quiet(bar.back(), (bc - 1) & 1u);  // the copies must land before the CTA leaves
          break;
        }
        for (int i = lane; i < (int)(tile_bytes / 16); i += 32)
          __stcg(reinterpret_cast<float4*>(blk) + i, make_float4(0.f, 0.f, 0.f, 0.f));
        __syncwarp();
        if (lane == 0) atomicExch(cnt + wt, 0u);
      }
    }
    if (kGlu && own) {  // y = act(factor * gate) * (factor * up)
      auto out = [&](int slot, int j) {
        float g = lds_f32(pb + 4u * ((uint32_t)slot * kPStride + (uint32_t)j));
        float u = lds_f32(pb + 4u * ((uint32_t)slot * kPStride + (uint32_t)(kTileRows / 2 + j)));
        if (has_gs) {
          g = __fmul_rn(g, factor);
          u = __fmul_rn(u, factor);
        }
        return glu_act(p.glu_act, g) * u;
      };
      if ((ncols & 7) == 0) {
        for (int idx = lane; idx < M * (kTileRows / 16); idx += 32) {
          const int slot = idx / (kTileRows / 16), j8 = (idx % (kTileRows / 16)) * 8;
          if (j8 >= rows) continue;
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = out(slot, j8 + i);
          store_out8(a.y, p.x_is_bf16, (int64_t)slot * ncols + n0 + j8, v);
        }
      } else {
        for (int idx = lane; idx < M * (kTileRows / 2); idx += 32) {
          const int slot = idx / (kTileRows / 2), j = idx % (kTileRows / 2);
          if (j < rows) store_out(a.y, p.x_is_bf16, (int64_t)slot * ncols + n0 + j, out(slot, j));
        }
      }
    } else if (own) {  // write y = factor * sum for the tile's rows
      if ((a.N & 7) == 0) {
        // eight outputs (16 bytes) per store: a warp's narrow 2-byte stores
        // cost about as much each as a wide one
        for (int idx = lane; idx < M * (kTileRows / 8); idx += 32) {
          const int slot = idx / (kTileRows / 8), r8 = (idx % (kTileRows / 8)) * 8;
          if (r8 >= rows) continue;
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[i] = lds_f32(pb + 4u * ((uint32_t)slot * kPStride + (uint32_t)(r8 + i)));
            if (has_gs) v[i] = __fmul_rn(v[i], factor);
          }
          store_out8(a.y, p.x_is_bf16, (kGrp ? yrow[slot] : (int64_t)slot) * a.N + n0 + r8, v);
        }
      } else {
        for (int idx = lane; idx < M * kTileRows; idx += 32) {
          const int slot = idx / kTileRows, row = idx % kTileRows;
          if (row >= rows) continue;
          const float v = lds_f32(pb + 4u * ((uint32_t)slot * kPStride + (uint32_t)row));
          store_out(a.y, p.x_is_bf16, (kGrp ? yrow[slot] : (int64_t)slot) * a.N + n0 + row,
                    has_gs ? __fmul_rn(v, factor) : v);
        }
      }
    }
    // The buffer is free: its bulk add completed before the count and its
    // read-back landed.
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.pempty(b));
  }
}

// ---- expert groups (GatherQMM) ----
//
// A GatherQMM call with at most one row per CTA is run as expert groups:
// rows are grouped by expert index, in row order, at most kGroupRows to a
// group (one MMA token tile), and group ids follow the order in which the
// experts first appear. Every CTA derives the same grouping from the index
// arrays and serves one group: group g owns CTAs [g C / G, (g + 1) C / G) of
// the C in the grid (G <= R <= C, so every group has one), which split its
// expert's weight plane exactly as a dense call splits its plane. Each
// expert's weights are then streamed once per group instead of once per row.
constexpr int kGroupRows = 8;
constexpr uint32_t kNoExpert = 0xFFFFFFFFu;

struct GroupInfo {
  int G;       // groups in the call
  int expert;  // this CTA's group: expert index,
  int n;       // rows (1 .. kGroupRows),
  int gs, gi;  // CTAs serving it and this CTA's index among them,
  int wsbase;  // first of its workspace blocks
};

// Grouping, by all kT threads of the CTA; `scratch` holds 16 R bytes of
// shared memory. A row whose expert index is >= E or whose activation index
// is >= B belongs to no group: it is written as zeros, by CTA (row mod C).
// On return (after a barrier) info->G is set; when it is non-zero, info's
// other fields and yrow / xrow (output and activation row of each token slot)
// are written but not yet visible to other threads. info->n must be zero and
// visible on entry.
template <int kT>
__device__ void group_rows(const QmvArgs& a, uint8_t* scratch, int64_t* yrow, int64_t* xrow, GroupInfo* info) {
  const int R = (int)a.R, tid = (int)threadIdx.x, C = (int)gridDim.x, bid = (int)blockIdx.x;
  uint32_t* key = reinterpret_cast<uint32_t*>(scratch);  // expert of each row, or kNoExpert
  int* rank = reinterpret_cast<int*>(key + R);           // rows of the same expert before it
  int* lead = rank + R;                                  // first row of its expert
  int* base = lead + R;                                  // on a first row: the expert's first group id
  for (int t = tid; t < R; t += kT) {
    // batched weights: consecutive runs of rows_per_expert rows per expert
    const uint32_t e = a.rows_per_expert > 0 ? (uint32_t)(t / a.rows_per_expert) : __ldg(a.rhs + t);
    const uint32_t xr = a.lhs ? __ldg(a.lhs + t) : (uint32_t)t;
    key[t] = (int64_t)e < a.E && (int64_t)xr < a.B ? e : kNoExpert;
  }
  __syncthreads();
  for (int t = tid; t < R; t += kT) {
    const uint32_t e = key[t];
    int rk = 0, total = 0, ld = t;
    if (e != kNoExpert) {
      for (int j = 0; j < R; ++j) {
        const bool same = key[j] == e;
        total += same ? 1 : 0;
        if (same && j < t) {
          if (rk == 0) ld = j;
          ++rk;
        }
      }
    }
    rank[t] = rk;
    lead[t] = ld;
    base[t] = e != kNoExpert && rk == 0 ? (total + kGroupRows - 1) / kGroupRows : 0;
  }
  __syncthreads();
  if (tid < 32) {  // exclusive prefix sum over rows of the groups each expert needs
    const int per = (R + 31) / 32, lo = tid * per, hi = min(R, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += base[i];
    int inc = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, off);
      if (tid >= off) inc += v;
    }
    int run = inc - sum;
    for (int i = lo; i < hi; ++i) {
      const int v = base[i];
      base[i] = run;
      run += v;
    }
    if (tid == 31) info->G = inc;
  }
  __syncthreads();
  for (int t = bid; t < R; t += C) {  // rows without a group: exact +0.0
    if (key[t] != kNoExpert) continue;
    uint16_t* yr = static_cast<uint16_t*>(a.y) + (int64_t)t * a.N;
    if ((a.N & 7) == 0)
      for (int64_t i = tid; i < a.N / 8; i += kT) reinterpret_cast<uint4*>(yr)[i] = make_uint4(0, 0, 0, 0);
    else
      for (int64_t i = tid; i < a.N; i += kT) yr[i] = 0;
  }
  const int G = info->G;
  if (G == 0) return;
  const int g = (int)(((int64_t)(bid + 1) * G - 1) / C);  // the g with g C / G <= bid < (g + 1) C / G
  const int s0 = (int)((int64_t)g * C / G), s1 = (int)((int64_t)(g + 1) * C / G);
  for (int t = tid; t < R; t += kT) {
    const uint32_t e = key[t];
    if (e == kNoExpert || base[lead[t]] + rank[t] / kGroupRows != g) continue;
    const int slot = rank[t] % kGroupRows;
    yrow[slot] = t;
    xrow[slot] = a.lhs ? (int64_t)__ldg(a.lhs + t) : (int64_t)t;
    if (slot == 0) info->expert = (int)e;
    atomicAdd(&info->n, 1);
  }
  if (tid == 0) {
    info->gs = s1 - s0;
    info->gi = bid - s0;
    info->wsbase = s0;
  }
}

// Dynamic shared memory: [1024-aligned] word stages | scale blocks | partial
// buffers | barriers, abort flag | slot table | bf16 scale table, zero block |
// staged activations.
size_t stream_smem_bytes(const SPlan& p) {
  const size_t pbuf = (size_t)2 * p.pslots * kPStride * 4;
  const size_t xs = (((size_t)p.M * p.xs_stride * 2) + 15) & ~(size_t)15;
  return 1024 + (size_t)p.stages * kWBox + 2 * kSBox + pbuf + kBarBytes + 16 + 256 + 1024 + 512 + 64 + xs;
}

template <int MT, int RT, bool kGrp, bool kGlu = false>
__global__ void __launch_bounds__(Geo<RT>::kThreads, 1)
qmv_stream_kernel(const QmvArgs a, const SPlan p, float* __restrict__ acc, uint32_t* __restrict__ cnt,
                  const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  const uint32_t wst = base;                       // stages x 32 KB (1024-aligned)
  const uint32_t sst = wst + p.stages * kWBox;     // 2 x 16 KB
  const uint32_t pbuf = sst + 2 * kSBox;           // 2 partial buffers
  const uint32_t pbuf_bytes = (uint32_t)(p.pslots * kPStride * 4);
  const Bars bar{pbuf + 2 * pbuf_bytes, p.stages};
  uint8_t* after_bars = bp + (bar.base - base) + kBarBytes;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(after_bars);
  int64_t* s_yrow = reinterpret_cast<int64_t*>(after_bars + 16);  // expert group: output row of each token slot
  int64_t* s_xrow = s_yrow + 16;                                     // and its activation row
  uint32_t* lut = reinterpret_cast<uint32_t*>(after_bars + 16 + 256);
  const uint32_t lut_bf = smem_addr(lut);
  // 512 zero bytes stand in for the activations of absent token slots; they
  // sit 64 bytes (mod 128) before the staged rows so that a lane reading them
  // and a lane reading row 0 in the same phase use different banks.
  const uint32_t zero_base = lut_bf + 1024;
  const uint32_t xs_base = zero_base + 512 + 64;
  __shared__ Corr s_corr[kMaxCorr];
  __shared__ int s_ncorr;
  __shared__ GroupInfo s_ginfo;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(bar.full(s), 1);     // producer arrive + TMA bytes
      mbar_init(bar.empty(s), Geo<RT>::kCW);  // one arrive per consumer warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.sfull(b), 1);
      mbar_init(bar.sempty(b), Geo<RT>::kCW);
      mbar_init(bar.pfull(b), Geo<RT>::kCW * 32);  // every consumer lane
      mbar_init(bar.pempty(b), 1);
    }
    mbar_init(bar.back(), 1);
    *abort_flag = 0;
    s_ncorr = 0;
    s_ginfo.n = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x == Geo<RT>::kProducer * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&smap)) : "memory");
  }
  if (threadIdx.x < 256) lut[threadIdx.x] = e4m3_to_bf16x2_bcast_x2p112(threadIdx.x);
  if (threadIdx.x < 128) lut[256 + threadIdx.x] = 0u;  // the zero block
  // Launched with launch overlap on, this grid may start while the previous
  // kernel on the stream finishes: the weight planes are streamed at once
  // (the caller guarantees no running kernel writes them); activations,
  // outputs and the workspace are touched only after griddepcontrol.wait.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();

  // A dense call: CTA b serves K group b / gs. An expert group: the CTA's
  // plan is the host's with the group's rows and CTA count.
  SPlan q = p;
  int grp = 0, gi = 0, expert = 0, wsbase = 0;
  if (kGrp) {
    // The indices may come from the kernel before: group after it completes,
    // in word stage 0, which the producer fills only afterwards.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    group_rows<Geo<RT>::kThreads>(a, bp, s_yrow, s_xrow, &s_ginfo);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (s_ginfo.G == 0) return;
    q.M = s_ginfo.n;
    q.gs = s_ginfo.gs;
    gi = s_ginfo.gi;
    expert = s_ginfo.expert;
    wsbase = s_ginfo.wsbase;
  } else {
    grp = blockIdx.x / p.gs;
    gi = blockIdx.x % p.gs;
  }
  const Work wk = Work::of(q, gi);

  if (warp == Geo<RT>::kProducer) {
    if ((threadIdx.x & 31) == 0) {
      ProdState pst;
      produce<kGrp, kGlu>(q, grp, wk, &wmap, &smap, wst, sst, bar, abort_flag, expert, pst, q.stages);
      drain_copies(pst, bar, q.stages);
    }
    return;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == Geo<RT>::kEpilogue) {
    FinState fst;
    finish<kGrp, kGlu>(a, q, wk, pbuf, pbuf_bytes, bar, abort_flag, acc, cnt, expert, wsbase, s_yrow, fst);
    return;
  }
  // Consumers: stage the activation columns this CTA visits (named barrier
  // 1, 512 threads), then stream.
  const XRun run = x_run(q, wk);
  const int mode = stage_run<Geo<RT>::kCW * 32, kGrp>(a, q, grp * q.ncg, run, xs_base, s_corr, &s_ncorr, s_xrow);
  ConsState cst;
  if (mode == 2)
    consume<__nv_bfloat16, MT, RT>(q, grp, wk, run, wst, sst, pbuf, pbuf_bytes, bar, abort_flag, xs_base, zero_base,
                                   lut_bf, s_corr, 0, cst, q.stages);
  else
    consume<__half, MT, RT>(q, grp, wk, run, wst, sst, pbuf, pbuf_bytes, bar, abort_flag, xs_base, zero_base, lut_bf,
                            s_corr, mode == 1 ? s_ncorr : 0, cst, q.stages);
}

// ---- a sequence of decode calls in one launch ----
//
// The calls of a decode step (the projections of a layer, at one or several
// token counts) run back to back in one persistent launch: each CTA walks its
// share of call 0's plane, then of call 1's, and so on, through one ring of
// word stages and one set of barriers. The producer streams call i + 1's
// weights while the consumers finish call i and the epilogue warp finishes
// call i's split tiles, so what a single call pays at its start (barrier
// set-up, the first TMA round trip, the ring filling) and at its end (the
// split-tile reduction, the last stores) is paid once per launch. A call may
// read outputs of earlier calls of the launch: its consumers then wait
// (bounded) until every CTA has finished every earlier call, which needs all
// CTAs resident at once (a cooperative launch); the producer keeps streaming
// its weights meanwhile.
constexpr int kSeqMaxCalls = 32;
// Largest grid whose CTAs the host reassigns per call (one byte per CTA).
constexpr int kSeqMaxGrid = 256;

struct SeqCall {
  CUtensorMap wmap, smap;  // first: 64-byte aligned
  QmvArgs a;
  SPlan p;
  int64_t ws_block;  // first workspace block (256-row tile) of this call
  int depends;       // wait for every earlier call before reading x
  // CTA b takes share pos[b] of this call's split (shares >= S * gs have no
  // work): the host deals the heavier shares of each call to the CTAs with
  // the least work so far, so that the per-call rounding of the split does
  // not pile up on the same CTAs. Identity when `permuted` is 0.
  int permuted;
  uint8_t pos[kSeqMaxGrid];
};
struct SeqArgs {
  SeqCall call[kSeqMaxCalls];
  int ncalls;
  int stages;    // word stages in the ring (all calls)
  int pslots;    // token slots of a partial buffer (8 or 16)
  int signal;    // some call depends on earlier ones: count finished calls
  int64_t done;  // counter words: done[c] at cnt[done + c], then the exit count
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait by one thread until *ctr >= target (release by the CTAs that
// counted in, acquire here); false once the limit passes (abort flag set,
// error code 28 recorded) or another warp has aborted.
__device__ bool wait_count(const uint32_t* ctr, uint32_t target, volatile int* abort_flag) {
  const uint64_t t0 = gtimer();
  for (;;) {
    if (ld_acquire_u32(ctr) >= target) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicCAS(&g_stream_error, 0, 28);
      return false;
    }
    __nanosleep(64);
  }
}

__device__ __forceinline__ int share_of(const SeqCall& C, int b) { return C.permuted ? (int)C.pos[b] : b; }

// Asks L2 for this CTA's 1/C share of a call's activations x (M K 16-bit
// values, contiguous; a multiple of 512 bytes), so that when the consumers
// stage the call they read L2 instead of waiting behind the weight stream in
// HBM.
__device__ __forceinline__ void prefetch_x_share(const QmvArgs& a, int b, int C) {
  const uint64_t bytes = (uint64_t)a.R * (uint64_t)a.K * 2u;
  const uint64_t share = ((bytes + (uint64_t)C - 1) / (uint64_t)C + 15u) & ~(uint64_t)15u;
  const uint64_t start = (uint64_t)b * share;
  if (start >= bytes) return;
  const uint64_t len = bytes - start < share ? bytes - start : share;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char*>(a.x) + start),
               "r"((uint32_t)len)
               : "memory");
}

// Dynamic shared memory of the sequence kernel: the single-call layout with
// a common ring depth, partial buffers of pslots token slots and room for the
// largest staged activation slice of any call.
size_t seq_smem_bytes(int stages, int pslots, size_t xs) {
  const size_t pbuf = (size_t)2 * pslots * kPStride * 4;
  return 1024 + (size_t)stages * kWBox + 2 * kSBox + pbuf + kBarBytes + 16 + 256 + 1024 + 512 + 64 +
         ((xs + 15) & ~(size_t)15);
}

__global__ void __launch_bounds__(Geo<1>::kThreads, 1)
qmv_seq_kernel(const __grid_constant__ SeqArgs sa, float* __restrict__ acc, uint32_t* __restrict__ cnt) {
  using G = Geo<1>;
  constexpr int kN = G::kCW * 32;  // consumer threads
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  const int stages = sa.stages;
  const uint32_t wst = base;
  const uint32_t sst = wst + stages * kWBox;
  const uint32_t pbuf = sst + 2 * kSBox;
  const uint32_t pbuf_bytes = (uint32_t)(sa.pslots * kPStride * 4);
  const Bars bar{pbuf + 2 * pbuf_bytes, stages};
  uint8_t* after_bars = bp + (bar.base - base) + kBarBytes;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(after_bars);
  uint32_t* lut = reinterpret_cast<uint32_t*>(after_bars + 16 + 256);
  const uint32_t lut_bf = smem_addr(lut);
  const uint32_t zero_base = lut_bf + 1024;
  const uint32_t xs_base = zero_base + 512 + 64;
  __shared__ Corr s_corr[kMaxCorr];
  __shared__ int s_ncorr;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < stages; ++st) {
      mbar_init(bar.full(st), 1);
      mbar_init(bar.empty(st), G::kCW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.sfull(b), 1);
      mbar_init(bar.sempty(b), G::kCW);
      mbar_init(bar.pfull(b), G::kCW * 32);
      mbar_init(bar.pempty(b), 1);
    }
    mbar_init(bar.back(), 1);
    *abort_flag = 0;
    s_ncorr = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == G::kProducer && lane == 0)
    for (int c = 0; c < sa.ncalls; ++c) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&sa.call[c].wmap)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&sa.call[c].smap)) : "memory");
    }
  if (threadIdx.x < 256) lut[threadIdx.x] = e4m3_to_bf16x2_bcast_x2p112(threadIdx.x);
  if (threadIdx.x < 128) lut[256 + threadIdx.x] = 0u;  // the zero block
  // With launch overlap the weights stream at once; activations, outputs and
  // the workspace are touched only after griddepcontrol.wait.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();

  const int b = (int)blockIdx.x;
  if (warp == G::kProducer) {
    if (lane == 0) {
      ProdState pst;
      for (int c = 0; c < sa.ncalls; ++c) {
        const SeqCall& C = sa.call[c];
        const int bc = share_of(C, b);
        if (bc >= C.p.S * C.p.gs) continue;
        // the consumers are still a ring's depth behind, on the previous call
        if (c > 0 && !C.depends) prefetch_x_share(C.a, b, (int)gridDim.x);
        if (!produce<false, false>(C.p, bc / C.p.gs, Work::of(C.p, bc % C.p.gs), &C.wmap, &C.smap, wst, sst, bar,
                                   abort_flag, 0, pst, stages))
          break;
      }
      drain_copies(pst, bar, stages);
    }
    return;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == G::kEpilogue) {
    FinState fst;
    for (int c = 0; c < sa.ncalls; ++c) {
      const SeqCall& C = sa.call[c];
      const int bc = share_of(C, b);
      if (bc < C.p.S * C.p.gs)
        finish<false, false>(C.a, C.p, Work::of(C.p, bc % C.p.gs), pbuf, pbuf_bytes, bar, abort_flag,
                             acc + C.ws_block * (int64_t)(kAccSlots * kTileRows), cnt + C.ws_block, 0, 0, nullptr,
                             fst);
      if (sa.signal) {  // this CTA has written all it writes of calls 0..c
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(cnt + sa.done + c, 1u);
      }
    }
    if (sa.signal && lane == 0) {
      // The last CTA out returns the counters to zero for the next launch
      // (every CTA has passed all its waits before it counts out).
      __threadfence();
      if (atomicAdd(cnt + sa.done + sa.ncalls, 1u) == gridDim.x - 1) {
        for (int c = 0; c < sa.ncalls; ++c) atomicExch(cnt + sa.done + c, 0u);
        atomicExch(cnt + sa.done + sa.ncalls, 0u);
      }
    }
    return;
  }
  // Consumers: per call, stage its activation columns (after the previous
  // call's last chunk, and after the calls it depends on have finished
  // everywhere), then stream.
  ConsState cst;
  bool staged = false;
  for (int c = 0; c < sa.ncalls; ++c) {
    const SeqCall& C = sa.call[c];
    const int bc = share_of(C, b);
    if (bc >= C.p.S * C.p.gs) continue;
    const int grp = bc / C.p.gs;
    const Work wk = Work::of(C.p, bc % C.p.gs);
    if (staged) {  // every consumer is done with the previous activations
      sync_all<kN>();
      if (threadIdx.x == 0) s_ncorr = 0;
      sync_all<kN>();
    }
    staged = true;
    if (C.depends) {
      if (threadIdx.x == 0) wait_count(cnt + sa.done + c - 1, gridDim.x, abort_flag);
      sync_all<kN>();
    }
    const XRun run = x_run(C.p, wk);
    const int mode = stage_run<kN, false, true>(C.a, C.p, grp * C.p.ncg, run, xs_base, s_corr, &s_ncorr, nullptr);
    const int ncorr = mode == 1 ? s_ncorr : 0;
    if (C.p.M > 8) {
      if (mode == 2)
        consume<__nv_bfloat16, 2, 1>(C.p, grp, wk, run, wst, sst, pbuf, pbuf_bytes, bar, abort_flag, xs_base,
                                     zero_base, lut_bf, s_corr, 0, cst, stages);
      else
        consume<__half, 2, 1>(C.p, grp, wk, run, wst, sst, pbuf, pbuf_bytes, bar, abort_flag, xs_base, zero_base,
                              lut_bf, s_corr, ncorr, cst, stages);
    } else {
      if (mode == 2)
        consume<__nv_bfloat16, 1, 1>(C.p, grp, wk, run, wst, sst, pbuf, pbuf_bytes, bar, abort_flag, xs_base,
                                     zero_base, lut_bf, s_corr, 0, cst, stages);
      else
        consume<__half, 1, 1>(C.p, grp, wk, run, wst, sst, pbuf, pbuf_bytes, bar, abort_flag, xs_base, zero_base,
                              lut_bf, s_corr, ncorr, cst, stages);
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// ---- workspace: one per (device, stream), grown on demand ----
struct Ws {
  float* acc = nullptr;
  uint32_t* cnt = nullptr;
  int64_t acc_floats = 0, cnt_words = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, Ws> g_ws;
std::vector<void*> g_ws_retired;  // replaced buffers, freed by nvfp4_shutdown

// Zeroes device memory on a library-owned stream and waits for it, so the
// clearing is never part of the caller's stream or of a graph capture.
cudaError_t zero_now(void* ptr, size_t bytes) {
  cudaStream_t z = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&z, cudaStreamNonBlocking);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(ptr, 0, bytes, z);
  const cudaError_t e2 = cudaStreamSynchronize(z);
  cudaStreamDestroy(z);
  return e != cudaSuccess ? e : e2;
}

// The workspace of (dev, st), allocated (zeroed) or grown on first need. A
// stream being captured into a graph (torch.cuda.graph captures on a stream
// of its own) gets its workspace with the thread's capture mode relaxed for
// the allocation, the way a stream-ordered allocator does it; the buffer is
// ready before the graph is ever replayed.
cudaError_t get_workspace(int dev, cudaStream_t st, int64_t nrt, Ws* out) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  Ws& w = g_ws[{dev, reinterpret_cast<uintptr_t>(st)}];
  const int64_t need_acc = nrt * kTileRows * kAccSlots, need_cnt = nrt;
  if (w.acc_floats < need_acc || w.cnt_words < need_cnt) {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaError_t e = cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) return e;
    const int64_t acc_n = need_acc > w.acc_floats * 2 ? need_acc : w.acc_floats * 2;
    const int64_t cnt_n = need_cnt > w.cnt_words * 2 ? need_cnt : w.cnt_words * 2;
    float* acc = nullptr;
    uint32_t* cnt = nullptr;
    e = cudaMalloc(&acc, (size_t)acc_n * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&cnt, (size_t)cnt_n * sizeof(uint32_t));
    if (e == cudaSuccess) e = zero_now(acc, (size_t)acc_n * sizeof(float));
    if (e == cudaSuccess) e = zero_now(cnt, (size_t)cnt_n * sizeof(uint32_t));
    cudaStreamCaptureMode back = mode;
    cudaThreadExchangeStreamCaptureMode(&back);
    if (e != cudaSuccess) {
      cudaFree(acc);
      cudaFree(cnt);
      return e;
    }
    if (w.acc) g_ws_retired.push_back(w.acc);
    if (w.cnt) g_ws_retired.push_back(w.cnt);
    w.acc = acc;
    w.cnt = cnt;
    w.acc_floats = acc_n;
    w.cnt_words = cnt_n;
  }
  *out = w;
  return cudaSuccess;
}

int sms_of(int dev) {
  int sms = 152;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

// Plan: for each ring depth (4, else 3 stages) the fewest K groups whose
// activation slice fits next to the ring; the depth with fewer groups wins
// (fewer groups means fewer row tiles finished through the workspace), ties
// go to the deeper ring. CTAs per group fill the SMs.
bool make_plan(SPlan& p, int sms, int64_t max_dyn) {
  const int mt = p.M > 8 ? 2 : 1;
  p.pslots = 8 * mt;
  bool found = false;
  SPlan best{};
  for (int stages = kMaxStages; stages >= 3; --stages) {
    for (int S = 1; S <= p.nc && S <= sms; ++S) {
      if (p.nc % S) continue;
      SPlan q = p;
      q.stages = stages;
      q.S = S;
      q.ncg = p.nc / S;
      const int64_t tg = q.nrt * q.ncg;
      const int64_t per = sms / S;
      q.gs = (int)(per < tg ? per : tg);
      if (q.gs < 1) continue;
      // a CTA with whole rows stages the group's chunks; otherwise its run
      const int64_t run = (tg + q.gs - 1) / q.gs;
      q.xs_chunks = q.nrt / q.gs >= 1 || run >= q.ncg ? q.ncg : (int)run;
      q.xs_stride = q.xs_chunks * kChunkCols + 32;
      if ((int64_t)stream_smem_bytes(q) > max_dyn) continue;
      if (!found || q.S < best.S) best = q;
      found = true;
      break;
    }
  }
  if (found) p = best;
  return found;
}

// TMA descriptors of a weight plane and its scale plane (words: 256-row x
// 128-byte boxes, 128-byte swizzle; scales: 256-row x 64-byte boxes, 64-byte
// swizzle). Encoding costs host time on every call, and decode-step weights
// are the same few planes call after call, so the pair is kept per (planes,
// shape). With `experts` the maps are 3-D over all E planes ([E, N, K], box
// depth 1), so that a box never runs into the next expert's rows.
// box_rows: 256 (a row tile per box), or 128 for a GLU tile's two halves.
cudaError_t plane_maps(const QmvArgs& a, CUtensorMap* wmap, CUtensorMap* smap, bool experts = false,
                       cuuint32_t box_rows = kTileRows) {
  using Key = std::tuple<const void*, const void*, int64_t, int64_t, int64_t, cuuint32_t>;
  struct Maps {
    CUtensorMap w, s;
  };
  static std::mutex mu;
  static std::map<Key, Maps> cache;
  const Key key{a.w, a.scales, a.N, a.K, experts ? a.E : 0, box_rows};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *wmap = it->second.w;
      *smap = it->second.s;
      return cudaSuccess;
    }
  }
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint32_t rank = experts ? 3 : 2;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)(a.K / 8), (cuuint64_t)a.N, (cuuint64_t)a.E};
    const cuuint64_t strides[2] = {(cuuint64_t)(a.K / 2), (cuuint64_t)(a.K / 2) * (cuuint64_t)a.N};
    const cuuint32_t box[3] = {kChunkWords, box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, rank, const_cast<uint32_t*>(a.w), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)(a.K / 16), (cuuint64_t)a.N, (cuuint64_t)a.E};
    const cuuint64_t strides[2] = {(cuuint64_t)(a.K / 16), (cuuint64_t)(a.K / 16) * (cuuint64_t)a.N};
    const cuuint32_t box[3] = {kSChunks * 16, box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<uint8_t*>(a.scales), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 1024) cache.clear();  // bound the table (weights are few; this never triggers in practice)
  cache[key] = Maps{*wmap, *smap};
  return cudaSuccess;
}

// The launch plan of a decode call, made once per (device, shape, M) and
// cached; cudaErrorInvalidConfiguration when no plan fits the SM's shared
// memory. `out` may be null (a check only).
template <int MT, int RT, bool kGlu = false>
cudaError_t stream_plan(const QmvArgs& a, int xdt, int dev, SPlan* out) {
  auto kern = qmv_stream_kernel<MT, RT, false, kGlu>;
  using Key = std::tuple<int, int64_t, int64_t, int64_t, int, int>;
  static std::mutex mu;
  static std::map<Key, SPlan> cache;
  static std::map<int, int64_t> max_dyn_of_dev;
  std::lock_guard<std::mutex> lock(mu);
  const Key key{dev, a.N, a.K, a.R, xdt, a.glu_act};
  auto it = cache.find(key);
  if (it != cache.end()) {
    if (out) *out = it->second;
    return cudaSuccess;
  }
  auto md = max_dyn_of_dev.find(dev);
  int64_t max_dyn;
  if (md == max_dyn_of_dev.end()) {
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    max_dyn = optin - (int64_t)fa.sharedSizeBytes;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_dyn)) != cudaSuccess)
      return e;
    max_dyn_of_dev[dev] = max_dyn;
  } else {
    max_dyn = md->second;
  }
  SPlan p{};
  p.M = (int)a.R;
  p.nc = (int)(a.K / kChunkCols);
  p.nrt = kGlu ? (a.glu_cols + kTileRows / 2 - 1) / (kTileRows / 2) : (a.N + kTileRows - 1) / kTileRows;
  p.x_is_bf16 = xdt == kBF16;
  p.glu_cols = a.glu_cols;
  p.glu_act = a.glu_act;
  if (!make_plan(p, sms_of(dev), max_dyn)) return cudaErrorInvalidConfiguration;
  p.wait_ns = kWaitLimitNs;
  p.withhold = 0;
  cache[key] = p;
  if (out) *out = p;
  return cudaSuccess;
}

template <int MT, int RT, bool kGlu = false>
cudaError_t launch_mt(const QmvArgs& a, int xdt, cudaStream_t st, const Ws* given = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  SPlan p{};
  if ((e = stream_plan<MT, RT, kGlu>(a, xdt, dev, &p)) != cudaSuccess) return e;
  // tests of the bounded waits: a shorter limit, and a withheld stage release
  if (const int us = option(kOptWaitLimitUs)) p.wait_ns = (uint64_t)us * 1000u;
  p.withhold = option(kOptTestWithhold);
  Ws ws;
  if (given)
    ws = *given;
  else if ((e = get_workspace(dev, st, p.nrt, &ws)) != cudaSuccess)
    return e;
  CUtensorMap wmap, smap;
  if ((e = plane_maps(a, &wmap, &smap, false, kGlu ? kTileRows / 2 : kTileRows)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.S * p.gs), 1, 1);
  cfg.blockDim = dim3(Geo<RT>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = stream_smem_bytes(p);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_overlap() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, qmv_stream_kernel<MT, RT, false, kGlu>, a, p, ws.acc, ws.cnt, wmap, smap);
}

// One launch for up to 16 token rows: eight token slots per MMA tile (MT),
// and RT weight row tiles per consumer warp (RT = 2 shares each activation
// fragment between two row tiles; the NVFP4_OPT_QMV_ROW_TILES option
// overrides the choice).
cudaError_t launch_rows(const QmvArgs& a, int xdt, cudaStream_t st, const Ws* ws) {
  int rt = a.R > 8 ? 2 : 1;
  const int forced = option(kOptQmvRowTiles);
  if (forced == 1 || forced == 2) rt = forced;
  if (a.R > 8) return rt == 2 ? launch_mt<2, 2>(a, xdt, st, ws) : launch_mt<2, 1>(a, xdt, st, ws);
  return rt == 2 ? launch_mt<1, 2>(a, xdt, st, ws) : launch_mt<1, 1>(a, xdt, st, ws);
}

// Expert-group launch (GatherQMM): one K group, so that a CTA stages the
// whole activation rows of its group once; the deepest ring that fits next to
// them. Shared-memory limit per device, looked up once.
bool group_plan(const QmvArgs& a, int xdt, int dev, SPlan* out) {
  static std::mutex mu;
  static std::map<int, int64_t> max_dyn_of_dev;
  int64_t max_dyn = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto md = max_dyn_of_dev.find(dev);
    if (md == max_dyn_of_dev.end()) {
      auto kern = qmv_stream_kernel<1, 1, true>;
      int optin = 0;
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return false;
      max_dyn = optin - (int64_t)fa.sharedSizeBytes;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_dyn) != cudaSuccess)
        return false;
      max_dyn_of_dev[dev] = max_dyn;
    } else {
      max_dyn = md->second;
    }
  }
  SPlan p{};
  p.M = kGroupRows;
  p.pslots = kGroupRows;
  p.nc = (int)(a.K / kChunkCols);
  p.nrt = (a.N + kTileRows - 1) / kTileRows;
  p.x_is_bf16 = xdt == kBF16;
  p.S = 1;
  p.ncg = p.nc;
  p.gs = 1;  // per group, set by each CTA
  p.xs_chunks = p.nc;
  p.xs_stride = p.nc * kChunkCols + 32;
  p.wait_ns = kWaitLimitNs;
  p.withhold = 0;
  for (int stages = kMaxStages; stages >= 3; --stages) {
    p.stages = stages;
    if ((int64_t)stream_smem_bytes(p) <= max_dyn) {
      *out = p;
      return true;
    }
  }
  return false;
}

}  // namespace

bool qmv_group_supported(const QmvArgs& a, int xdt) {
  if (option(kOptGatherGroup) == 0) return false;
  if (xdt == kF32 || (a.rhs == nullptr && a.rows_per_expert <= 0) || a.R < 1 || a.K % kChunkCols != 0 || a.K <= 0 ||
      a.N <= 0 ||
      a.N >= (1ll << 31) || a.K / kChunkCols > 4096 || a.E < 1 || a.E >= (1ll << 31))
    return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  SPlan p;
  return a.R <= sms_of(dev) && group_plan(a, xdt, dev, &p);
}

// One CTA per SM; every CTA groups the rows itself (no planning launch).
cudaError_t launch_qmv_group(const QmvArgs& a, int xdt, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  SPlan p;
  const int C = sms_of(dev);
  if (a.R > C || !group_plan(a, xdt, dev, &p)) return cudaErrorInvalidConfiguration;
  Ws ws;
  if ((e = get_workspace(dev, st, C, &ws)) != cudaSuccess) return e;
  CUtensorMap wmap, smap;
  if ((e = plane_maps(a, &wmap, &smap, true)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, 1, 1);
  cfg.blockDim = dim3(Geo<1>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = stream_smem_bytes(p);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_overlap() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, qmv_stream_kernel<1, 1, true>, a, p, ws.acc, ws.cnt, wmap, smap);
}

bool qmv_stream_supported(const QmvArgs& a, int xdt) {
  return xdt != kF32 && a.rhs == nullptr && a.lhs == nullptr && a.E == 1 && a.R >= 1 && a.K % kChunkCols == 0 &&
         a.K > 0 && a.N > 0 && a.N < (1ll << 31) && a.K / kChunkCols <= 4096;
}

// More than 16 token rows run as consecutive launches of 16 rows each (the
// weights are streamed once per launch).
cudaError_t launch_qmv_stream(const QmvArgs& a, int xdt, cudaStream_t st) {
  for (int64_t r0 = 0; r0 < a.R; r0 += 16) {
    QmvArgs b = a;
    b.R = b.B = a.R - r0 < 16 ? a.R - r0 : 16;
    b.x = static_cast<const uint16_t*>(a.x) + r0 * a.K;
    b.y = static_cast<uint16_t*>(a.y) + r0 * a.N;
    const cudaError_t e = launch_rows(b, xdt, st, nullptr);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Fused gate/up: 16 token rows per launch as for a plain call; y has
// glu_cols columns.
cudaError_t launch_qmv_stream_glu(const QmvArgs& a, int xdt, cudaStream_t st) {
  for (int64_t r0 = 0; r0 < a.R; r0 += 16) {
    QmvArgs b = a;
    b.R = b.B = a.R - r0 < 16 ? a.R - r0 : 16;
    b.x = static_cast<const uint16_t*>(a.x) + r0 * a.K;
    b.y = static_cast<uint16_t*>(a.y) + r0 * a.glu_cols;
    const cudaError_t e = b.R > 8 ? launch_mt<2, 2, true>(b, xdt, st) : launch_mt<1, 1, true>(b, xdt, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---- host side of the call sequence ----
namespace {

// A call's plan for a given ring depth: the fewest K groups whose staged
// activation slice fits in `xs_budget` bytes (as make_plan); false if none.
bool seq_call_plan(SPlan& p, int sms, int64_t xs_budget) {
  for (int S = 1; S <= p.nc && S <= sms; ++S) {
    if (p.nc % S) continue;
    SPlan q = p;
    q.S = S;
    q.ncg = p.nc / S;
    const int64_t tg = q.nrt * q.ncg;
    const int64_t per = sms / S;
    q.gs = (int)(per < tg ? per : tg);
    if (q.gs < 1) continue;
    const int64_t run = (tg + q.gs - 1) / q.gs;
    q.xs_chunks = q.nrt / q.gs >= 1 || run >= q.ncg ? q.ncg : (int)run;
    q.xs_stride = q.xs_chunks * kChunkCols + 32;
    if ((int64_t)q.M * q.xs_stride * 2 > xs_budget) continue;
    p = q;
    return true;
  }
  return false;
}

int64_t seq_max_dyn(int dev) {
  static std::mutex mu;
  static std::map<int, int64_t> of_dev;
  std::lock_guard<std::mutex> lock(mu);
  auto it = of_dev.find(dev);
  if (it != of_dev.end()) return it->second;
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, qmv_seq_kernel) != cudaSuccess) return -1;
  const int64_t max_dyn = optin - (int64_t)fa.sharedSizeBytes;
  if (cudaFuncSetAttribute(qmv_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_dyn) != cudaSuccess)
    return -1;
  of_dev[dev] = max_dyn;
  return max_dyn;
}

}  // namespace

bool qmv_seq_call_supported(const QmvArgs& a, int xdt) {
  return xdt != kF32 && a.rhs == nullptr && a.lhs == nullptr && a.E == 1 && a.R >= 1 && a.R <= 16 &&
         a.K % kChunkCols == 0 && a.K > 0 && a.N > 0 && a.N < (1ll << 31) && a.K / kChunkCols <= 4096;
}

cudaError_t launch_qmv_seq(const QmvArgs* calls, const int* depends, int n, int xdt, cudaStream_t st) {
  if (n < 1 || n > kSeqMaxCalls) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int64_t max_dyn = seq_max_dyn(dev);
  if (max_dyn < 0) return cudaErrorInvalidConfiguration;
  const int sms = sms_of(dev);
  static_assert(sizeof(SeqArgs) + 2 * sizeof(void*) <= 32764, "kernel parameters exceed the launch limit");
  auto sa = std::make_unique<SeqArgs>();
  std::memset(sa.get(), 0, sizeof(SeqArgs));
  int pslots = 8;
  bool any_dep = false;
  for (int c = 0; c < n; ++c) {
    if (calls[c].R > 8) pslots = 16;
    any_dep = any_dep || (c > 0 && depends[c]);
  }
  // One ring depth for every call: the depth whose calls need the fewest K
  // groups in all (fewer row tiles finished through the workspace), ties to
  // the deeper ring; each call takes the fewest groups its slice allows.
  int best_stages = 0;
  int64_t best_groups = 0;
  std::vector<SPlan> best(n), cur(n);
  for (int stages = kMaxStages; stages >= 3; --stages) {
    const int64_t budget = max_dyn - (int64_t)seq_smem_bytes(stages, pslots, 0);
    if (budget < 0) continue;
    int64_t groups = 0;
    bool ok = true;
    for (int c = 0; c < n && ok; ++c) {
      SPlan p{};
      p.M = (int)calls[c].R;
      p.nc = (int)(calls[c].K / kChunkCols);
      p.nrt = (calls[c].N + kTileRows - 1) / kTileRows;
      p.x_is_bf16 = xdt == kBF16;
      p.stages = stages;
      p.pslots = pslots;
      ok = seq_call_plan(p, sms, budget);
      cur[c] = p;
      groups += p.S;
    }
    if (ok && (best_stages == 0 || groups < best_groups)) {
      best_stages = stages;
      best_groups = groups;
      best = cur;
    }
  }
  if (best_stages == 0) return cudaErrorInvalidConfiguration;
  int64_t blocks = 0;
  size_t xs = 0;
  for (int c = 0; c < n; ++c) {
    SeqCall& C = sa->call[c];
    C.a = calls[c];
    C.p = best[c];
    C.p.wait_ns = kWaitLimitNs;
    C.p.withhold = 0;
    C.ws_block = blocks;
    C.depends = c > 0 && depends[c] ? 1 : 0;
    blocks += C.p.nrt;
    xs = std::max(xs, (size_t)C.p.M * C.p.xs_stride * 2);
    if ((e = plane_maps(C.a, &C.wmap, &C.smap)) != cudaSuccess) return e;
  }
  // Deal each call's shares: the heaviest (most chunks, a 16-token chunk
  // counted 1.3 times) to the CTAs with the least work so far.
  if (sms <= kSeqMaxGrid) {
    std::vector<double> load(sms, 0.0);
    std::vector<int> by_load(sms), by_share(sms);
    std::vector<double> share(sms);
    for (int c = 0; c < n; ++c) {
      SeqCall& C = sa->call[c];
      const SPlan& p = C.p;
      const double wgt = p.M > 8 ? 1.3 : 1.0;
      const int64_t W = p.nrt / p.gs, rest = (p.nrt - W * p.gs) * p.ncg;
      for (int i = 0; i < sms; ++i) {
        if (i >= p.S * p.gs) {
          share[i] = 0.0;
          continue;
        }
        const int64_t gi = i % p.gs;
        share[i] = wgt * (double)(W * p.ncg + rest * (gi + 1) / p.gs - rest * gi / p.gs);
      }
      for (int i = 0; i < sms; ++i) by_load[i] = by_share[i] = i;
      std::stable_sort(by_load.begin(), by_load.end(), [&](int x, int y) { return load[x] < load[y]; });
      std::stable_sort(by_share.begin(), by_share.end(), [&](int x, int y) { return share[x] > share[y]; });
      for (int k = 0; k < sms; ++k) {
        C.pos[by_load[k]] = (uint8_t)by_share[k];
        load[by_load[k]] += share[by_share[k]];
      }
      C.permuted = 1;
    }
  }
  sa->ncalls = n;
  sa->stages = best_stages;
  sa->pslots = pslots;
  sa->signal = any_dep ? 1 : 0;
  sa->done = blocks;  // the counter words after the tile counters
  Ws ws;
  // blocks tile blocks of sums and counters, plus n + 1 counter words
  if ((e = get_workspace(dev, st, blocks + kSeqMaxCalls + 1, &ws)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms, 1, 1);
  cfg.blockDim = dim3(Geo<1>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = seq_smem_bytes(best_stages, pslots, xs);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (any_dep) {
    // the dependent waits need every CTA resident at once
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = any_dep || launch_overlap() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, qmv_seq_kernel, *sa, ws.acc, ws.cnt);
}

int read_stream_error() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_stream_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(int));
    // An aborted kernel may have left partial sums and counts behind: clear
    // every workspace once all work has finished.
    cudaDeviceSynchronize();
    std::lock_guard<std::mutex> lock(g_ws_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_ws) {
      cudaSetDevice(kv.first.first);
      cudaDeviceSynchronize();
      zero_now(kv.second.acc, (size_t)kv.second.acc_floats * sizeof(float));
      zero_now(kv.second.cnt, (size_t)kv.second.cnt_words * sizeof(uint32_t));
    }
    cudaSetDevice(cur);
  }
  return v;
}

// ---- allocation-free variant --------------------------------------------
//
// The same decode kernel, with its scratch (the split-tile sums and the tile
// counters) in a fixed array compiled into the library instead of a
// workspace from cudaMalloc. It serves callers that must not allocate device
// memory: a runtime whose memory is planned once at start-up, or code that
// runs while a CUDA graph is being captured in the strict mode, where an
// allocation would break the capture. The array costs every GPU that loads
// the library kNoAllocBytes until the process exits.
namespace {
constexpr int64_t kNoAllocAccFloats = (int64_t)kAccSlots * kNoAllocMaxRows;  // 4 MB of sums
constexpr int64_t kNoAllocCounters = kNoAllocMaxRows / kTileRows;           // one per 256-row tile
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocAccFloats + kNoAllocCounters];

struct NoAllocDev {
  float* base = nullptr;  // device address of g_noalloc_scratch on this device
  bool ready = false;
};
std::mutex g_noalloc_mu;
std::map<int, NoAllocDev> g_noalloc;

// Device address of the array on the current device (its host-side name is
// only a stand-in), looked up once per device.
cudaError_t noalloc_base(int dev, float** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDev& d = g_noalloc[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    d.base = static_cast<float*>(ptr);
    d.ready = true;
  }
  *out = d.base;
  return cudaSuccess;
}

// Whether the decode kernel has a launch plan for this shape (the plan the
// launch itself will use, cached the same way).
bool noalloc_plan_ok(const QmvArgs& a, int xdt, int dev) {
  if (a.R > 8) return stream_plan<2, 2>(a, xdt, dev, nullptr) == cudaSuccess;
  return stream_plan<1, 1>(a, xdt, dev, nullptr) == cudaSuccess;
}
}  // namespace

cudaError_t launch_qmv_stream_noalloc(const QmvArgs& a, int xdt, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // Resolve the launch plan first, so that a shape the kernel cannot take is
  // refused before anything is queued on the stream.
  if (!noalloc_plan_ok(a, xdt, dev)) return cudaErrorInvalidConfiguration;
  float* base = nullptr;
  if ((e = noalloc_base(dev, &base)) != cudaSuccess) return e;
  const int64_t nrt = (a.N + kTileRows - 1) / kTileRows;
  Ws ws;
  ws.acc = base;
  ws.cnt = reinterpret_cast<uint32_t*>(base + kNoAllocAccFloats);
  ws.acc_floats = kNoAllocAccFloats;
  ws.cnt_words = kNoAllocCounters;
  // Row tile r's sums are block r (16 slots x 256 floats), of which a call
  // with M token rows uses the first M slots: clear those and the tile
  // counters (a previous call may have been cut short and left them dirty).
  if ((e = cudaMemsetAsync(ws.cnt, 0, (size_t)nrt * sizeof(uint32_t), st)) != cudaSuccess) return e;
  if ((e = cudaMemset2DAsync(ws.acc, (size_t)kAccSlots * kTileRows * sizeof(float), 0,
                             (size_t)a.R * kTileRows * sizeof(float), (size_t)nrt, st)) != cudaSuccess)
    return e;
  return launch_rows(a, xdt, st, &ws);
}

void release_noalloc_addresses() {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  g_noalloc.clear();
}

void release_stream_workspaces() {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  for (auto& kv : g_ws) {
    cudaFree(kv.second.acc);
    cudaFree(kv.second.cnt);
  }
  g_ws.clear();
  for (void* ptr : g_ws_retired) cudaFree(ptr);
  g_ws_retired.clear();
}

}  // namespace nvfp4
