// Prefill-shape NVFP4 QuantizedMatmul on the 5th-generation tensor cores.
//
// y[m, n] = factor * sum_k x[m, k] * (fp4 * e4m3)[n, k] for large M (mlxcel PR
// #2629 "ROCm native NVFP4", Summary: prefill-size products take a dense GEMM
// route; the global scale multiplies each output once, after the sum).
//
// The pages' route dequantizes the whole plane and calls a vendor GEMM. Here
// the dequantization is fused into a persistent tcgen05 GEMM: the weights are
// read packed (9/16 byte per element) and expanded tile by tile in shared
// memory, so the dense plane never exists in HBM. The products fp4 * e4m3 are
// exact in bf16/f16, so the tensor core sees exactly the dequantized weights.
//
// Per CTA (one per SM), for a BM x BN output tile with BM = 128 * MH:
//   warp 0      TMA producer of the activation tiles x[BM x 64] (SW128), one
//               128-row box per M half
//   warp 1      MMA issuer: tcgen05.mma.cta_group::1.kind::f16, M=128 per M
//               half, N=BN, K=16; accumulators in TMEM
//   warp 2      TMEM allocator
//   warps 4..   epilogue, four warps per M half: tcgen05.ld 32x32b, global
//               factor, cast, store
//   last 8      weight producers: 128-bit loads of the packed words and scale
//               bytes (four to six k-blocks ahead in registers), exact
//               decode to bf16/f16, stores in the canonical K-major
//               128-byte-swizzled layout the MMA descriptor reads
// Every decoded weight tile feeds MH M=128 MMAs, so a 256-row tile (MH = 2)
// halves the decode work per flop, which is what bounds the bf16 route.
// Stages hand off through mbarriers; every wait is bounded and records an
// error code instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

__device__ int g_tc_error = 0;  // first error code recorded by a bounded wait

namespace {

constexpr int BK = 64;
constexpr uint32_t kHalfA = 128 * BK * 2;  // one 128-row activation box: 16 KB
constexpr uint32_t kRingBudget = 192 * 1024;
constexpr int kProducerWarps = 8;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpAlloc = 2, kWarpEpi0 = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Tile configuration: MH M halves of 128 rows, BN weight rows per tile.
template <int MH_, int BN_>
struct Cfg {
  static constexpr int MH = MH_, BN = BN_, BM = 128 * MH_;
  static constexpr uint32_t A_BYTES = MH_ * kHalfA;
  static constexpr uint32_t B_BYTES = BN_ * BK * 2;
  static constexpr int STAGES = (int)(kRingBudget / (A_BYTES + B_BYTES));
  static constexpr int ACC_BUFS = (int)kTmemCols / (MH_ * BN_) >= 2 ? 2 : 1;  // accumulator buffers in TMEM
  static constexpr int EPI_WARPS = 4 * MH_;
  static constexpr int kWarpProd0 = kWarpEpi0 + EPI_WARPS;
  static constexpr int THREADS = 32 * (kWarpProd0 + kProducerWarps);
  static constexpr int RPT = BN_ / 128;  // weight rows per producer thread
  static constexpr int PF = RPT == 1 ? 6 : 4;  // k-blocks of packed weights in flight per producer thread
  static constexpr int BAR_BYTES = 8 * (3 * STAGES + 2 * ACC_BUFS) + 16;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * (A_BYTES + B_BYTES) + BAR_BYTES;
  static_assert(STAGES >= 3, "ring too shallow");
  static_assert(ACC_BUFS * MH_ * BN_ <= (int)kTmemCols, "accumulators exceed TMEM");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct TcParams {
  const uint32_t* w;
  const uint8_t* scales;
  const float* gs;
  void* y;
  int64_t M, N, K;  // M = output rows (R for a gather)
  int num_m_tiles, num_tiles, num_kb, num_n_tiles;
  // Expert-batched gather (GatherQMM with rows sorted by expert): output row
  // r is x[lhs[r]] (x[r] without lhs) times expert rhs[r]'s weights.
  const uint32_t* lhs;
  const uint32_t* rhs;
  int64_t B;    // activation rows
  int E;        // experts
  // Stream-K launches (qmm_tc_sk_kernel): tiles [0, dp_tiles) are dealt
  // whole, round robin; the k-block iterations of tiles [dp_tiles, dp_tiles +
  // sk_tiles) are divided evenly over the CTAs. A tile shared by several CTAs
  // is summed in ws (BM x BN floats per tile, column-major so that a warp's
  // 32 rows of one column are 128 contiguous bytes; sk_tiles of them) and
  // finished by the CTA whose k-blocks complete ws_cnt[tile - dp_tiles]; both
  // are left zeroed.
  int dp_tiles, sk_tiles;
  float* ws;
  uint32_t* ws_cnt;
  // Fused gate/up (qmm_tc_kernel with kGlu): the plane holds 2 * glu_cols
  // rows (gate, then up); weight tile nt stands for gate rows [128 nt, 128 nt
  // + 128) and the matching up rows, and y ([M, glu_cols]) gets act(gate) *
  // up. glu_act: 1 SiLU, 2 GELU (tanh form).
  int64_t glu_cols;
  int glu_act;
  // bf16 activations served by the f16 kernel (rows_to_f16_kernel, output
  // type bf16): row m of the f16 activations is the bf16 row times 1 /
  // row_scale[m], so each sum is multiplied by row_scale[m] (a power of two).
  const float* row_scale = nullptr;
};

// Output bits of one value in the output type. The f16 kernels that serve
// bf16 rows (output type bf16) scale each row's sums by row_scale; the others
// have no scaling code at all.
template <typename T, typename TO>
__device__ __forceinline__ float row_factor(const TcParams& p, int64_t m) {
  if constexpr (std::is_same<T, TO>::value) {
    return 1.0f;
  } else {
    return __ldg(p.row_scale + m);  // an exact power of two
  }
}
template <typename TO>
__device__ __forceinline__ uint32_t out_bits(float v) {
  const TO t = Dt<TO>::from_f32(v);
  return *reinterpret_cast<const uint16_t*>(&t);
}

// One output tile: expert, weight tile, first output row and row count.
struct Tile {
  int e, nt, rows;
  int64_t m0;
};

// Shared-memory tables of the gather mode: seg[e] = first row of expert e
// (seg[E] = first row whose expert is out of range), pre[e] = tiles of the
// experts before e (pre[E] = all tiles).
constexpr int kGatherMaxE = 1024;
constexpr int kGatherSamples = 4096;
constexpr size_t kGatherSmem = (size_t)kGatherSamples * 4 + 2 * (size_t)(kGatherMaxE + 1) * 4 + 16;

template <bool GATHER, int BM>
__device__ __forceinline__ Tile tile_of(const TcParams& p, int t, const int* seg, const int* pre) {
  Tile r;
  if (!GATHER) {
    const int mt = t % p.num_m_tiles;
    r.e = 0;
    r.nt = t / p.num_m_tiles;
    r.m0 = (int64_t)mt * BM;
    const int64_t left = p.M - r.m0;
    r.rows = left < BM ? (int)left : BM;
    return r;
  }
  // largest e with pre[e] <= t; experts without rows have no tiles, so the
  // search never lands on one
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= t) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int cnt = seg[e + 1] - seg[e];
  const int mtiles = (cnt + BM - 1) / BM;
  const int rem = t - pre[e];
  r.e = e;
  r.nt = rem / mtiles;  // m tiles fastest: consecutive tiles share a weight tile
  r.m0 = seg[e] + (int64_t)(rem % mtiles) * BM;
  const int64_t left = seg[e + 1] - r.m0;
  r.rows = left < BM ? (int)left : BM;
  return r;
}

// A run of k-blocks [kb0, kb1) of one tile.
struct Unit {
  int tile, kb0, kb1;
};

// A CTA's units, in the order every role walks them: its share of the
// stream-K iterations (tile-major, k-blocks fastest, cut at tile boundaries),
// then its data-parallel tiles (blockIdx.x, + gridDim.x, ...). Split tiles come
// first so that finishing them overlaps the whole tiles that follow.
struct Sched {
  int i_dp, n_dp, num_kb, dp;
  int64_t it, it_end;
  __device__ __forceinline__ void init(int dp_tiles, int sk_tiles, int kbs) {
    dp = dp_tiles;
    num_kb = kbs;
    n_dp = (int)blockIdx.x < dp_tiles ? (dp_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    i_dp = 0;
    const int64_t I = (int64_t)sk_tiles * kbs;
    it = I * blockIdx.x / gridDim.x;
    it_end = I * (blockIdx.x + 1) / gridDim.x;
  }
  // k-blocks this CTA will process in all
  __device__ __forceinline__ int64_t total() const { return (int64_t)(n_dp - i_dp) * num_kb + (it_end - it); }
  __device__ __forceinline__ bool next(Unit& u) {
    if (it < it_end) {
      const int64_t t = it / num_kb;
      u.tile = dp + (int)t;
      u.kb0 = (int)(it - t * num_kb);
      const int64_t left = it_end - it;
      u.kb1 = left < (int64_t)(num_kb - u.kb0) ? u.kb0 + (int)left : num_kb;
      it += u.kb1 - u.kb0;
      return true;
    }
    if (i_dp >= n_dp) return false;
    u.tile = (int)blockIdx.x + i_dp * (int)gridDim.x;
    u.kb0 = 0;
    u.kb1 = num_kb;
    ++i_dp;
    return true;
  }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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
// Bounded wait: false (and the abort flag set) after kWaitLimitNs, or as soon
// as another role has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int code) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(&g_tc_error, 0, code);
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128
// bytes, eight-row groups 1024 bytes apart (stride byte offset), descriptor
// version 1 (bits 46-48), swizzle mode 2 (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor for kind::f16: f32 accumulator, A/B bf16 or f16,
// both K-major, N = BN, M = 128.
template <bool BF16, int BN>
__host__ __device__ constexpr uint32_t make_idesc() {
  return (1u << 4) | ((BF16 ? 1u : 0u) << 7) | ((BF16 ? 1u : 0u) << 10) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

#define NVFP4_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : NVFP4_R8(0), NVFP4_R8(8), NVFP4_R8(16), NVFP4_R8(24)
      : "r"(taddr));
}
#undef NVFP4_R8
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- producer of decoded weights

template <int RPT>
struct WTask {
  uint4 w[RPT];      // packed words 4h..4h+3 of the k-block for rows r + 128 i
  uint32_t s[RPT];   // the four scale bytes of the k-block for those rows
};

struct WCursor {
  int tile, kb;
  bool done;
  int e, nt;  // expert and weight tile of `tile`
};

template <bool GATHER, int BM>
__device__ __forceinline__ void w_seek(WCursor& cur, const TcParams& p, int num_tiles, const int* seg, const int* pre) {
  cur.done = cur.tile >= num_tiles;
  if (!cur.done) {
    const Tile t = tile_of<GATHER, BM>(p, cur.tile, seg, pre);
    cur.e = t.e;
    cur.nt = t.nt;
  }
}

template <int BN, bool kGlu = false, int RPT, typename Cur>
__device__ __forceinline__ void w_load(WTask<RPT>& t, const Cur& cur, const TcParams& p, int r, int h) {
  if (cur.done) return;
  const int64_t kwords = p.K / 8, kgroups = p.K / 16;
  const uint32_t* w = p.w + (int64_t)cur.e * p.N * kwords;
  const uint8_t* sc = p.scales + (int64_t)cur.e * p.N * kgroups;
  const int64_t kw = (int64_t)cur.kb * 8 + 4 * h;  // first of this task's four words
  const bool kok = kw < kwords;                     // K % 32 == 0 keeps the four words together
  const int64_t g4 = (int64_t)cur.kb * 4;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    // GLU: the first 128 rows of the tile are gate rows, the next 128 the up
    // rows of the same outputs
    const int64_t n = kGlu ? (int64_t)cur.nt * 128 + r + (i ? p.glu_cols : 0) : (int64_t)cur.nt * BN + r + 128 * i;
    const bool ok = kok && (kGlu ? (int64_t)cur.nt * 128 + r < p.glu_cols : n < p.N);
    t.w[i] = ok ? __ldg(reinterpret_cast<const uint4*>(w + n * kwords + kw)) : make_uint4(0, 0, 0, 0);
    if (kgroups % 4 == 0) {
      t.s[i] = ok ? __ldg(reinterpret_cast<const uint32_t*>(sc + n * kgroups + g4)) : 0u;
    } else {
      uint32_t v = 0;
      for (int j = 0; j < 4; ++j)
        if (ok && g4 + j < kgroups) v |= (uint32_t)sc[n * kgroups + g4 + j] << (8 * j);
      t.s[i] = v;
    }
  }
}

template <bool GATHER, int BM>
__device__ __forceinline__ void w_advance(WCursor& cur, const TcParams& p, int num_tiles, const int* seg,
                                          const int* pre) {
  if (++cur.kb >= p.num_kb) {
    cur.kb = 0;
    cur.tile += gridDim.x;
    w_seek<GATHER, BM>(cur, p, num_tiles, seg, pre);
  }
}

// Decode one row's four words (columns 32h..32h+31 of the k-block) and store
// them as four 16-byte chunks of the swizzled row.
template <typename T>
__device__ __forceinline__ void w_store_row(uint32_t stage_base, int row, int h, const uint4& w, uint32_t sbytes) {
  const uint32_t sc0 = Dt<T>::scale((sbytes >> (16 * h)) & 0xFF);
  const uint32_t sc1 = Dt<T>::scale((sbytes >> (16 * h + 8)) & 0xFF);
  const uint32_t rbase = stage_base + (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u;
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t o[4];
    Dt<T>::decode(ws[i], i < 2 ? sc0 : sc1, o);
    const uint32_t chunk = (uint32_t)(4 * h + i) ^ (uint32_t)(row & 7);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(rbase + chunk * 16u), "r"(o[0]), "r"(o[1]),
                 "r"(o[2]), "r"(o[3])
                 : "memory");
  }
}

template <typename T, typename C, bool GATHER, bool kGlu = false>
__device__ void producer_role(const TcParams& p, uint32_t sB, uint32_t bars, volatile int* abort_flag, int num_tiles,
                              const int* seg, const int* pre) {
  constexpr int STAGES = C::STAGES, RPT = C::RPT, BM = C::BM;
  const int pid = threadIdx.x - C::kWarpProd0 * 32;  // 0..255
  const int r = pid >> 1, h = pid & 1;               // rows r + 128 i, words 4h..4h+3 of the k-block
  const int lane = threadIdx.x & 31;
  WCursor ld{(int)blockIdx.x, 0, true, 0, 0};
  w_seek<GATHER, BM>(ld, p, num_tiles, seg, pre);
  // PF k-blocks of packed weights in flight per thread (registers), so that
  // the L2 latency of the loads is covered by PF - 1 blocks of decoding.
  constexpr int PF = C::PF;
  WTask<RPT> buf[PF];
#pragma unroll
  for (int j = 0; j < PF - 1; ++j) {
    w_load<C::BN, kGlu>(buf[j], ld, p, r, h);
    w_advance<GATHER, BM>(ld, p, num_tiles, seg, pre);
  }
  uint32_t u = 0;
  const int total = ((num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) * p.num_kb;
  auto consume = [&](const WTask<RPT>& t) -> bool {
    const int s = (int)(u % STAGES);
    const uint32_t ph = (u / STAGES) & 1;
    if (!wait_bar_warp(bars + 8 * (2 * STAGES + s), ph ^ 1, abort_flag, 3, &g_tc_error)) return false;  // stage empty
    const uint32_t stage = sB + (uint32_t)s * C::B_BYTES;
#pragma unroll
    for (int i = 0; i < RPT; ++i) w_store_row<T>(stage, r + 128 * i, h, t.w[i], t.s[i]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (STAGES + s));  // fullB
    ++u;
    return true;
  };
  // the ring of buffers is indexed by compile-time positions only (unrolled),
  // so it stays in registers
  for (int i = 0; i < total; i += PF) {
#pragma unroll
    for (int j = 0; j < PF; ++j) {
      if (i + j >= total) return;
      w_load<C::BN, kGlu>(buf[(j + PF - 1) % PF], ld, p, r, h);
      w_advance<GATHER, BM>(ld, p, num_tiles, seg, pre);
      if (!consume(buf[j])) return;
    }
  }
}

// ---------------------------------------------------------------- non-transposed weights
//
// A non-transposed plane is quantized along the output axis (mlx PR #2629,
// Changes during review: the K-multiple-of-16 rule applies to N when the
// weight is not transposed): word w[k][j] holds outputs 8j..8j+7 of input k,
// one scale byte per 16 outputs of an input, and y = x @ dequantize(w). The
// tensor cores still take K-major weight tiles, so the producer transposes
// while it decodes: producer warp v takes inputs 8v..8v+7 of the k-block and
// lane j word column j of the tile; per output it then holds eight
// consecutive k values, which is one 16-byte chunk of the output's swizzled
// B row. Lane j starts at output (j & 7) of its word (the word is rotated by
// that many nibbles before decoding), so the eight lanes of a quarter-warp
// store to eight different 16-byte bank groups.

struct WTaskNT {
  uint32_t w[8];  // inputs k0..k0+7 of the lane's word column
  uint32_t s;     // scale bytes 4 (lane & 3) .. + 3 of the tile's 16 for input k0 + (lane >> 2)
};

// Loaded values are only stored in registers here (no arithmetic on them),
// so issuing the loads of later k-blocks never waits for their data.
template <typename Cur>
__device__ __forceinline__ void w_load_nt(WTaskNT& t, const Cur& cur, const TcParams& p, int v, int j) {
  if (cur.done) return;
  const int64_t nwords = p.N / 8, ngroups = p.N / 16;
  const int64_t col = (int64_t)cur.nt * 32 + j;
  const bool cok = col < nwords;
  const int64_t k0 = (int64_t)cur.kb * BK + 8 * v;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int64_t k = k0 + kk;
    t.w[kk] = cok && k < p.K ? __ldg(p.w + k * nwords + col) : 0u;  // inputs past K decode to +0
  }
  const int64_t ks = k0 + (j >> 2), g0 = (int64_t)cur.nt * 16 + 4 * (j & 3);
  uint32_t sv = 0;
  if (ks < p.K) {
    const uint8_t* row = p.scales + ks * ngroups;
    if ((ngroups & 3) == 0) {
      if (g0 < ngroups) sv = __ldg(reinterpret_cast<const uint32_t*>(row + g0));
    } else {
      for (int q = 0; q < 4; ++q)
        if (g0 + q < ngroups) sv |= (uint32_t)__ldg(row + g0 + q) << (8 * q);
    }
  }
  t.s = sv;
}

// lut: shared-memory table of Dt<T>::scale for the 256 scale bytes (a lane
// converts eight scale bytes per k-block, one per input row).
template <typename T>
__device__ __forceinline__ void w_store_nt(uint32_t stage_base, int v, int j, const WTaskNT& t, uint32_t lut) {
  const int rot = j & 7;
  uint32_t o[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    // the scale byte of the lane's 16-output block (j / 2) for input kk
    const uint32_t quad = __shfl_sync(0xffffffffu, t.s, kk * 4 + (j >> 3));
    const uint32_t sb = (quad >> (8 * ((j >> 1) & 3))) & 0xFFu;
    uint32_t sc;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc) : "r"(lut + 4u * sb));
    Dt<T>::decode(__funnelshift_r(t.w[kk], t.w[kk], 4 * rot), sc, o[kk]);
  }
  const uint32_t rows = stage_base + (uint32_t)j * 1024u;  // B rows 8j..8j+7
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t oc = (uint32_t)((c + rot) & 7);  // output 8j + oc of the tile
    const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = __byte_perm(o[2 * i][c >> 1], o[2 * i + 1][c >> 1], sel);
    const uint32_t addr = rows + oc * 128u + (((uint32_t)v ^ oc) * 16u);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                 : "memory");
  }
}

template <typename T, typename C>
__device__ void producer_role_nt(const TcParams& p, uint32_t sB, uint32_t bars, volatile int* abort_flag,
                                 int num_tiles, uint32_t lut) {
  static_assert(C::BN == 256 && kProducerWarps * 8 == BK, "one word column per lane, eight inputs per warp");
  // one k-block of words loaded ahead (nine registers): on GB300 this ran
  // faster than two or three ahead (M = 8192 on [5376, 21504]: 1683 us
  // against 2131 and 1880), whose registers the 640-thread CTA cannot spare
  constexpr int STAGES = C::STAGES, PF = 2, BM = C::BM;
  const int v = (int)(threadIdx.x >> 5) - C::kWarpProd0;
  const int j = threadIdx.x & 31;
  WCursor ld{(int)blockIdx.x, 0, true, 0, 0};
  w_seek<false, BM>(ld, p, num_tiles, nullptr, nullptr);
  WTaskNT buf[PF];
#pragma unroll
  for (int i = 0; i < PF - 1; ++i) {
    w_load_nt(buf[i], ld, p, v, j);
    w_advance<false, BM>(ld, p, num_tiles, nullptr, nullptr);
  }
  uint32_t u = 0;
  const int total = ((num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) * p.num_kb;
  auto consume = [&](const WTaskNT& t) -> bool {
    const int s = (int)(u % STAGES);
    const uint32_t ph = (u / STAGES) & 1;
    if (!wait_bar_warp(bars + 8 * (2 * STAGES + s), ph ^ 1, abort_flag, 3, &g_tc_error)) return false;  // stage empty
    w_store_nt<T>(sB + (uint32_t)s * C::B_BYTES, v, j, t, lut);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (j == 0) mbar_arrive(bars + 8 * (STAGES + s));  // fullB
    ++u;
    return true;
  };
  for (int i = 0; i < total; i += PF) {
#pragma unroll
    for (int q = 0; q < PF; ++q) {
      if (i + q >= total) return;
      w_load_nt(buf[(q + PF - 1) % PF], ld, p, v, j);
      w_advance<false, BM>(ld, p, num_tiles, nullptr, nullptr);
      if (!consume(buf[q])) return;
    }
  }
}

// ---------------------------------------------------------------- stream-K variants
//
// The stream-K kernel walks units (tile, k-block range) instead of whole
// tiles; its roles are kept apart from the whole-tile kernel's so that the
// latter compiles exactly as before (sharing them cost it 6% at M = 8192).

struct WCursorSK {
  Sched sc;
  Unit un;
  int kb;
  bool done;
  int e, nt;  // expert and weight tile of the current unit's tile
};

template <bool GATHER, int BM>
__device__ __forceinline__ void w_seek_sk(WCursorSK& cur, const TcParams& p, const int* seg, const int* pre) {
  cur.done = !cur.sc.next(cur.un);
  if (!cur.done) {
    cur.kb = cur.un.kb0;
    const Tile t = tile_of<GATHER, BM>(p, cur.un.tile, seg, pre);
    cur.e = t.e;
    cur.nt = t.nt;
  }
}

template <bool GATHER, int BM>
__device__ __forceinline__ void w_advance_sk(WCursorSK& cur, const TcParams& p, const int* seg, const int* pre) {
  if (!cur.done && ++cur.kb >= cur.un.kb1) w_seek_sk<GATHER, BM>(cur, p, seg, pre);
}

template <typename T, typename C, bool GATHER>
__device__ void producer_role_sk(const TcParams& p, uint32_t sB, uint32_t bars, volatile int* abort_flag, Sched sched,
                              const int* seg, const int* pre) {
  constexpr int STAGES = C::STAGES, RPT = C::RPT, BM = C::BM;
  const int pid = threadIdx.x - C::kWarpProd0 * 32;  // 0..255
  const int r = pid >> 1, h = pid & 1;               // rows r + 128 i, words 4h..4h+3 of the k-block
  const int lane = threadIdx.x & 31;
  WCursorSK ld;
  ld.sc = sched;
  const int64_t total = sched.total();
  w_seek_sk<GATHER, BM>(ld, p, seg, pre);
  // PF k-blocks of packed weights in flight per thread (registers), so that
  // the L2 latency of the loads is covered by PF - 1 blocks of decoding.
  constexpr int PF = C::PF;
  WTask<RPT> buf[PF];
#pragma unroll
  for (int j = 0; j < PF - 1; ++j) {
    w_load<C::BN>(buf[j], ld, p, r, h);
    w_advance_sk<GATHER, BM>(ld, p, seg, pre);
  }
  uint32_t u = 0;
  auto consume = [&](const WTask<RPT>& t) -> bool {
    const int s = (int)(u % STAGES);
    const uint32_t ph = (u / STAGES) & 1;
    if (!wait_bar_warp(bars + 8 * (2 * STAGES + s), ph ^ 1, abort_flag, 3, &g_tc_error)) return false;  // stage empty
    const uint32_t stage = sB + (uint32_t)s * C::B_BYTES;
#pragma unroll
    for (int i = 0; i < RPT; ++i) w_store_row<T>(stage, r + 128 * i, h, t.w[i], t.s[i]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (STAGES + s));  // fullB
    ++u;
    return true;
  };
  // the ring of buffers is indexed by compile-time positions only (unrolled),
  // so it stays in registers
  for (int64_t i = 0; i < total; i += PF) {
#pragma unroll
    for (int j = 0; j < PF; ++j) {
      if (i + j >= total) return;
      w_load<C::BN>(buf[(j + PF - 1) % PF], ld, p, r, h);
      w_advance_sk<GATHER, BM>(ld, p, seg, pre);
      if (!consume(buf[j])) return;
    }
  }
}

// Non-transposed weights in the stream-K kernel: the units of the stream-K
// schedule, the decode and transpose of producer_role_nt.
template <typename T, typename C>
__device__ void producer_role_sk_nt(const TcParams& p, uint32_t sB, uint32_t bars, volatile int* abort_flag,
                                    Sched sched, uint32_t lut) {
  static_assert(C::BN == 256 && kProducerWarps * 8 == BK, "one word column per lane, eight inputs per warp");
  constexpr int STAGES = C::STAGES, PF = 2, BM = C::BM;  // as in producer_role_nt
  const int v = (int)(threadIdx.x >> 5) - C::kWarpProd0;
  const int j = threadIdx.x & 31;
  WCursorSK ld;
  ld.sc = sched;
  const int64_t total = sched.total();
  w_seek_sk<false, BM>(ld, p, nullptr, nullptr);
  WTaskNT buf[PF];
#pragma unroll
  for (int i = 0; i < PF - 1; ++i) {
    w_load_nt(buf[i], ld, p, v, j);
    w_advance_sk<false, BM>(ld, p, nullptr, nullptr);
  }
  uint32_t u = 0;
  auto consume = [&](const WTaskNT& t) -> bool {
    const int s = (int)(u % STAGES);
    const uint32_t ph = (u / STAGES) & 1;
    if (!wait_bar_warp(bars + 8 * (2 * STAGES + s), ph ^ 1, abort_flag, 3, &g_tc_error)) return false;  // stage empty
    w_store_nt<T>(sB + (uint32_t)s * C::B_BYTES, v, j, t, lut);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (j == 0) mbar_arrive(bars + 8 * (STAGES + s));  // fullB
    ++u;
    return true;
  };
  for (int64_t i = 0; i < total; i += PF) {
#pragma unroll
    for (int q = 0; q < PF; ++q) {
      if (i + q >= total) return;
      w_load_nt(buf[(q + PF - 1) % PF], ld, p, v, j);
      w_advance_sk<false, BM>(ld, p, nullptr, nullptr);
      if (!consume(buf[q])) return;
    }
  }
}

// Gather mode: builds seg[] and pre[] from the expert indices (all threads of
// the CTA; ends with __syncthreads). A sample of every L-th index narrows each
// expert's lower-bound search to at most L rows of global memory. Indices
// that are not sorted still give non-decreasing segments covering every row
// below seg[E] exactly once, so no row is written twice or read out of range.
template <int BM>
__device__ void build_gather_tables(const TcParams& p, uint32_t* samp, int* seg, int* pre) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const int64_t R = p.M;
  const int64_t L = (R + kGatherSamples - 1) / kGatherSamples;  // >= 1
  const int ns = (int)((R + L - 1) / L);
  for (int j = tid; j < ns; j += nth) samp[j] = __ldg(p.rhs + (int64_t)j * L);
  __syncthreads();
  for (int e = tid; e <= p.E; e += nth) {
    const uint32_t ev = (uint32_t)e;
    int lo = 0, hi = ns;  // first sample >= e
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (samp[mid] < ev) lo = mid + 1; else hi = mid;
    }
    int64_t a = lo == 0 ? 0 : (int64_t)(lo - 1) * L + 1;
    int64_t b = lo == ns ? R : (int64_t)lo * L;
    while (a < b) {
      const int64_t mid = (a + b) >> 1;
      if (__ldg(p.rhs + mid) < ev) a = mid + 1; else b = mid;
    }
    seg[e] = (int)a;
  }
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    // non-decreasing segment starts (already so for sorted indices)
    const int n = p.E + 1, per = (n + 31) / 32, b = lane * per, en = min(b + per, n);
    int run = 0;
    for (int i = b; i < en; ++i) {
      run = max(run, seg[i]);
      seg[i] = run;
    }
    int m = run;
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, m, off);
      if (lane >= off) m = max(m, v);
    }
    int excl = __shfl_up_sync(0xffffffffu, m, 1);
    if (lane == 0) excl = 0;
    for (int i = b; i < en; ++i) seg[i] = max(seg[i], excl);
    __syncwarp();
    // tiles of each expert (row tiles times weight tiles), exclusive prefix sum
    const int ne = p.E, pe = (ne + 31) / 32, b2 = lane * pe, en2 = min(b2 + pe, ne);
    int sum = 0;
    for (int i = b2; i < en2; ++i) sum += ((seg[i + 1] - seg[i] + BM - 1) / BM) * p.num_n_tiles;
    int inc = sum;
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += v;
    }
    int base = inc - sum;
    for (int i = b2; i < en2; ++i) {
      pre[i] = base;
      base += ((seg[i + 1] - seg[i] + BM - 1) / BM) * p.num_n_tiles;
    }
    if (lane == 31) pre[ne] = inc;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- kernel

// TO: the output type (T, or bf16 when the f16 kernel serves bf16 rows).
template <typename T, typename C, bool GATHER, bool kGlu = false, bool kNT = false, typename TO = T>
__global__ void __launch_bounds__(C::THREADS, 1)
qmm_tc_kernel(const __grid_constant__ CUtensorMap xmap, const TcParams p) {
  constexpr int STAGES = C::STAGES, MH = C::MH, BN = C::BN, BM = C::BM, NBUF = C::ACC_BUFS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + STAGES * C::A_BYTES;
  const uint32_t bars = sB + STAGES * C::B_BYTES;
  // barriers: fullA[S] fullB[S] empty[S] accFull[NBUF] accEmpty[NBUF]
  uint32_t* holder =
      reinterpret_cast<uint32_t*>(base_ptr + STAGES * (C::A_BYTES + C::B_BYTES) + 8 * (3 * STAGES + 2 * NBUF));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(holder + 1);
  // gather tables follow the barrier block (16-byte aligned)
  uint32_t* samp = reinterpret_cast<uint32_t*>(base_ptr + C::SMEM - 1024);
  int* seg = reinterpret_cast<int*>(samp + kGatherSamples);
  int* pre = seg + (kGatherMaxE + 1);
  auto fullA = [&](int s) { return bars + 8 * s; };
  auto fullB = [&](int s) { return bars + 8 * (STAGES + s); };
  auto emptyB = [&](int s) { return bars + 8 * (2 * STAGES + s); };
  auto accFull = [&](int b) { return bars + 8 * (3 * STAGES + b); };
  auto accEmpty = [&](int b) { return bars + 8 * (3 * STAGES + NBUF + b); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(fullA(s), 1);
      mbar_init(fullB(s), kProducerWarps);
      mbar_init(emptyB(s), 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(accFull(b), 1);
      mbar_init(accEmpty(b), C::EPI_WARPS);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpTma && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
  if (warp == kWarpAlloc) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (GATHER) build_gather_tables<BM>(p, samp, seg, pre);  // ends with __syncthreads
  if constexpr (kNT) {  // the scale table of the non-transposed producer (1 KB past the barriers)
    if (threadIdx.x < 256) samp[threadIdx.x] = Dt<T>::scale(threadIdx.x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  const int num_tiles = GATHER ? pre[p.E] : p.num_tiles;
  const int my_tiles = (int)blockIdx.x < num_tiles
                           ? (num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                           : 0;

  if (warp == kWarpTma) {
    uint32_t u = 0;
    if (!GATHER) {
      if (lane == 0) {
        bool ok = true;
        for (int i = 0; i < my_tiles && ok; ++i) {
          const int tile = (int)blockIdx.x + i * (int)gridDim.x;
          const int m_tile = tile % p.num_m_tiles;
          for (int kb = 0; kb < p.num_kb; ++kb, ++u) {
            const int s = (int)(u % STAGES);
            const uint32_t ph = (u / STAGES) & 1;
            if (!wait_bar(emptyB(s), ph ^ 1, abort_flag, 1)) { ok = false; break; }
            mbar_arrive_tx(fullA(s), C::A_BYTES);
#pragma unroll
            for (int h = 0; h < MH; ++h)
              tma_load_2d(sA + (uint32_t)s * C::A_BYTES + (uint32_t)h * kHalfA, &xmap, kb * BK, m_tile * BM + 128 * h,
                          fullA(s));
          }
        }
      }
    } else {
      // The tile's activations are rows m0 .. m0 + rows - 1 of the mapped x:
      // one 128-row box per M half that holds rows of the tile (rows past
      // them belong to the next expert or lie beyond x; they are computed but
      // not stored).
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const Tile tl = tile_of<true, BM>(p, (int)blockIdx.x + i * (int)gridDim.x, seg, pre);
        const int mh = (tl.rows + 127) / 128;
        for (int kb = 0; kb < p.num_kb; ++kb, ++u) {
          const int s = (int)(u % STAGES);
          const uint32_t ph = (u / STAGES) & 1;
          if (!wait_bar_warp(emptyB(s), ph ^ 1, abort_flag, 1, &g_tc_error)) { ok = false; break; }
          if (lane == 0) {
            mbar_arrive_tx(fullA(s), (uint32_t)mh * kHalfA);
#pragma unroll
            for (int h = 0; h < MH; ++h)
              if (h < mh)
                tma_load_2d(sA + (uint32_t)s * C::A_BYTES + (uint32_t)h * kHalfA, &xmap, kb * BK,
                            (int)(tl.m0 + 128 * h), fullA(s));
          }
          __syncwarp();
        }
      }
    }
    // Leave no copy in flight: wait (bounded) for the last stages issued.
    if (lane == 0) {
      const uint32_t first = u > (uint32_t)STAGES ? u - STAGES : 0;
      for (uint32_t v = first; v < u; ++v) {
        const uint32_t limit_ph = (v / STAGES) & 1;
        const uint64_t t0 = gtimer();
        while (!mbar_try(fullA((int)(v % STAGES)), limit_ph) && gtimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc<std::is_same<T, __nv_bfloat16>::value, BN>();
      uint32_t u = 0;
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int b = i % NBUF;
        int mh = MH;  // M halves holding rows of the tile (a gather tile may fill one)
        if (GATHER) mh = (tile_of<true, BM>(p, (int)blockIdx.x + i * (int)gridDim.x, seg, pre).rows + 127) / 128;
        if (!wait_bar(accEmpty(b), ((i / NBUF) & 1) ^ 1, abort_flag, 4)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * MH * BN);
        for (int kb = 0; kb < p.num_kb; ++kb, ++u) {
          const int s = (int)(u % STAGES);
          const uint32_t ph = (u / STAGES) & 1;
          if (!wait_bar(fullA(s), ph, abort_flag, 5) || !wait_bar(fullB(s), ph, abort_flag, 6)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bd = sw128_desc(sB + (uint32_t)s * C::B_BYTES);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j)
#pragma unroll
            for (int h = 0; h < MH; ++h) {
              if (h >= mh) continue;
              const uint64_t ad = sw128_desc(sA + (uint32_t)s * C::A_BYTES + (uint32_t)h * kHalfA);
              umma_f16(d + (uint32_t)(h * BN), ad + (uint64_t)(2 * j), bd + (uint64_t)(2 * j), idesc, (kb | j) != 0);
            }
          umma_commit(emptyB(s));
        }
        if (ok) umma_commit(accFull(b));
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + C::EPI_WARPS) {
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int hm = (warp - kWarpEpi0) >> 2;  // M half it drains
    TO* y = static_cast<TO*>(p.y);
    if (GATHER) {
      // rows whose expert index is out of range (sorted last) are exact +0
      const int64_t z0 = seg[p.E];
      const int64_t total = (p.M - z0) * p.N;
      const int ethreads = 32 * C::EPI_WARPS, etid = threadIdx.x - 32 * kWarpEpi0;
      uint16_t* yz = reinterpret_cast<uint16_t*>(y) + z0 * p.N;
      for (int64_t i = (int64_t)blockIdx.x * ethreads + etid; i < total; i += (int64_t)gridDim.x * ethreads) yz[i] = 0;
    }
    for (int i = 0; i < my_tiles; ++i) {
      const Tile tl = tile_of<GATHER, BM>(p, (int)blockIdx.x + i * (int)gridDim.x, seg, pre);
      const int b = i % NBUF;
      if (!wait_bar_warp(accFull(b), (i / NBUF) & 1, abort_flag, 7, &g_tc_error)) break;
      tc_fence_after();
      const int rr = 128 * hm + 32 * q + lane;  // row within the tile
      const int64_t m = tl.m0 + rr;
      const bool live = rr < tl.rows;
      bool zero = false;
      if (GATHER && live) {
        const int64_t xr = p.lhs ? (int64_t)__ldg(p.lhs + m) : m;
        zero = xr >= p.B;
      }
      const float fac = global_factor(p.gs, tl.e);
      constexpr bool kRowScale = !std::is_same<T, TO>::value;
      const float rsc = kRowScale && live ? row_factor<T, TO>(p, m) : 1.0f;
      const int64_t n_base = (int64_t)tl.nt * BN;
      const uint32_t tcol = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * MH * BN + hm * BN);
      if constexpr (kGlu) {
        // columns [0, 128) hold gate sums, [128, 256) the matching up sums
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tcol + (uint32_t)(32 * c), g);
          tmem_ld32(tcol + (uint32_t)(BN / 2 + 32 * c), u);
          tmem_ld_wait();
          if (!live) continue;
          const int64_t n0 = (int64_t)tl.nt * (BN / 2) + 32 * c;
          if (n0 >= p.glu_cols) continue;
          uint32_t packed[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float o[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float gv = __uint_as_float(g[2 * k + e]), uv = __uint_as_float(u[2 * k + e]);
              if (kRowScale) {
                gv *= rsc;
                uv *= rsc;
              }
              if (p.gs) {
                gv = __fmul_rn(gv, fac);
                uv = __fmul_rn(uv, fac);
              }
              // SiLU: v sigmoid(v); GELU (tanh form): v sigmoid(2 sqrt(2/pi) (v + 0.044715 v^3))
              const float z = p.glu_act == 1 ? gv : 1.5957691216057308f * (gv + 0.044715f * gv * gv * gv);
              o[e] = __fdividef(gv, 1.0f + __expf(-z)) * uv;
            }
            packed[k] = out_bits<TO>(o[0]) | (out_bits<TO>(o[1]) << 16);
          }
          TO* dst = y + m * p.glu_cols + n0;
          if (n0 + 32 <= p.glu_cols && (p.glu_cols % 8) == 0) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              d4[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
          } else {
            uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
            for (int k = 0; k < 32 && n0 + k < p.glu_cols; ++k) d16[k] = (uint16_t)(packed[k >> 1] >> (16 * (k & 1)));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accEmpty(b));
        continue;
      }
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tcol + (uint32_t)(32 * c), r);
        tmem_ld_wait();
        if (!live) continue;
        const int64_t n0 = n_base + 32 * c;
        if (n0 >= p.N) continue;
        uint32_t packed[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float v0 = __uint_as_float(r[2 * k]), v1 = __uint_as_float(r[2 * k + 1]);
          if (kRowScale) {
            v0 *= rsc;
            v1 *= rsc;
          }
          if (p.gs) {
            v0 = __fmul_rn(v0, fac);
            v1 = __fmul_rn(v1, fac);
          }
          packed[k] = zero ? 0u : out_bits<TO>(v0) | (out_bits<TO>(v1) << 16);
        }
        TO* dst = y + m * p.N + n0;
        if (n0 + 32 <= p.N && (p.N % 8) == 0) {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            d4[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
        } else {
          uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
          for (int k = 0; k < 32 && n0 + k < p.N; ++k)
            d16[k] = (uint16_t)(packed[k >> 1] >> (16 * (k & 1)));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accEmpty(b));
    }
  } else if (warp >= C::kWarpProd0) {
    if constexpr (kNT)
      producer_role_nt<T, C>(p, sB, bars, abort_flag, num_tiles, smem_u32(samp));
    else
      producer_role<T, C, GATHER, kGlu>(p, sB, bars, abort_flag, num_tiles, seg, pre);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpAlloc) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// The stream-K kernel (dense launches of fewer than two waves of tiles): the
// same roles as qmm_tc_kernel, walking units (tile, k-block range), with the
// split-tile epilogue. Instantiated with GATHER = false and SK = true only.
template <typename T, typename C, bool GATHER, bool SK, bool kNT = false, typename TO = T>
__global__ void __launch_bounds__(C::THREADS, 1)
qmm_tc_sk_kernel(const __grid_constant__ CUtensorMap xmap, const TcParams p) {
  constexpr int STAGES = C::STAGES, MH = C::MH, BN = C::BN, BM = C::BM, NBUF = C::ACC_BUFS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + STAGES * C::A_BYTES;
  const uint32_t bars = sB + STAGES * C::B_BYTES;
  // barriers: fullA[S] fullB[S] empty[S] accFull[NBUF] accEmpty[NBUF]
  uint32_t* holder =
      reinterpret_cast<uint32_t*>(base_ptr + STAGES * (C::A_BYTES + C::B_BYTES) + 8 * (3 * STAGES + 2 * NBUF));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(holder + 1);
  // gather tables follow the barrier block (16-byte aligned)
  uint32_t* samp = reinterpret_cast<uint32_t*>(base_ptr + C::SMEM - 1024);
  int* seg = reinterpret_cast<int*>(samp + kGatherSamples);
  int* pre = seg + (kGatherMaxE + 1);
  auto fullA = [&](int s) { return bars + 8 * s; };
  auto fullB = [&](int s) { return bars + 8 * (STAGES + s); };
  auto emptyB = [&](int s) { return bars + 8 * (2 * STAGES + s); };
  auto accFull = [&](int b) { return bars + 8 * (3 * STAGES + b); };
  auto accEmpty = [&](int b) { return bars + 8 * (3 * STAGES + NBUF + b); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(fullA(s), 1);
      mbar_init(fullB(s), kProducerWarps);
      mbar_init(emptyB(s), 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(accFull(b), 1);
      mbar_init(accEmpty(b), C::EPI_WARPS);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpTma && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
  if (warp == kWarpAlloc) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (GATHER) build_gather_tables<BM>(p, samp, seg, pre);  // ends with __syncthreads
  if constexpr (kNT) {  // the scale table of the non-transposed producer (1 KB past the barriers)
    if (threadIdx.x < 256) samp[threadIdx.x] = Dt<T>::scale(threadIdx.x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  // Every role walks the same units; a gather's tiles (counted on the device)
  // are all dealt whole.
  Sched sched;
  if (GATHER)
    sched.init(pre[p.E], 0, p.num_kb);
  else
    sched.init(p.dp_tiles, p.sk_tiles, p.num_kb);
  __shared__ int s_fin;  // stream-K: this CTA completes the tile being finished

  if (warp == kWarpTma) {
    uint32_t u = 0;
    Unit un;
    if (!GATHER) {
      if (lane == 0) {
        bool ok = true;
        while (ok && sched.next(un)) {
          const int m_tile = un.tile % p.num_m_tiles;
          for (int kb = un.kb0; kb < un.kb1; ++kb, ++u) {
            const int s = (int)(u % STAGES);
            const uint32_t ph = (u / STAGES) & 1;
            if (!wait_bar(emptyB(s), ph ^ 1, abort_flag, 1)) { ok = false; break; }
            mbar_arrive_tx(fullA(s), C::A_BYTES);
#pragma unroll
            for (int h = 0; h < MH; ++h)
              tma_load_2d(sA + (uint32_t)s * C::A_BYTES + (uint32_t)h * kHalfA, &xmap, kb * BK, m_tile * BM + 128 * h,
                          fullA(s));
          }
        }
      }
    } else {
      // The tile's activations are rows m0 .. m0 + rows - 1 of the mapped x:
      // one 128-row box per M half that holds rows of the tile (rows past
      // them belong to the next expert or lie beyond x; they are computed but
      // not stored).
      bool ok = true;
      while (ok && sched.next(un)) {
        const Tile tl = tile_of<true, BM>(p, un.tile, seg, pre);
        const int mh = (tl.rows + 127) / 128;
        for (int kb = un.kb0; kb < un.kb1; ++kb, ++u) {
          const int s = (int)(u % STAGES);
          const uint32_t ph = (u / STAGES) & 1;
          if (!wait_bar_warp(emptyB(s), ph ^ 1, abort_flag, 1, &g_tc_error)) { ok = false; break; }
          if (lane == 0) {
            mbar_arrive_tx(fullA(s), (uint32_t)mh * kHalfA);
#pragma unroll
            for (int h = 0; h < MH; ++h)
              if (h < mh)
                tma_load_2d(sA + (uint32_t)s * C::A_BYTES + (uint32_t)h * kHalfA, &xmap, kb * BK,
                            (int)(tl.m0 + 128 * h), fullA(s));
          }
          __syncwarp();
        }
      }
    }
    // Leave no copy in flight: wait (bounded) for the last stages issued.
    if (lane == 0) {
      const uint32_t first = u > (uint32_t)STAGES ? u - STAGES : 0;
      for (uint32_t v = first; v < u; ++v) {
        const uint32_t limit_ph = (v / STAGES) & 1;
        const uint64_t t0 = gtimer();
        while (!mbar_try(fullA((int)(v % STAGES)), limit_ph) && gtimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc<std::is_same<T, __nv_bfloat16>::value, BN>();
      uint32_t u = 0;
      bool ok = true;
      Unit un;
      for (int i = 0; ok && sched.next(un); ++i) {
        const int b = i % NBUF;
        int mh = MH;  // M halves holding rows of the tile (a gather tile may fill one)
        if (GATHER) mh = (tile_of<true, BM>(p, un.tile, seg, pre).rows + 127) / 128;
        if (!wait_bar(accEmpty(b), ((i / NBUF) & 1) ^ 1, abort_flag, 4)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * MH * BN);
        for (int kb = un.kb0; kb < un.kb1; ++kb, ++u) {
          const int s = (int)(u % STAGES);
          const uint32_t ph = (u / STAGES) & 1;
          if (!wait_bar(fullA(s), ph, abort_flag, 5) || !wait_bar(fullB(s), ph, abort_flag, 6)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bd = sw128_desc(sB + (uint32_t)s * C::B_BYTES);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j)
#pragma unroll
            for (int h = 0; h < MH; ++h) {
              if (h >= mh) continue;
              const uint64_t ad = sw128_desc(sA + (uint32_t)s * C::A_BYTES + (uint32_t)h * kHalfA);
              umma_f16(d + (uint32_t)(h * BN), ad + (uint64_t)(2 * j), bd + (uint64_t)(2 * j), idesc,
                       ((kb - un.kb0) | j) != 0);
            }
          umma_commit(emptyB(s));
        }
        if (ok) umma_commit(accFull(b));
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + C::EPI_WARPS) {
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int hm = (warp - kWarpEpi0) >> 2;  // M half it drains
    const int etid = threadIdx.x - 32 * kWarpEpi0;
    TO* y = static_cast<TO*>(p.y);
    if (GATHER) {
      // rows whose expert index is out of range (sorted last) are exact +0
      const int64_t z0 = seg[p.E];
      const int64_t total = (p.M - z0) * p.N;
      const int ethreads = 32 * C::EPI_WARPS;
      uint16_t* yz = reinterpret_cast<uint16_t*>(y) + z0 * p.N;
      for (int64_t i = (int64_t)blockIdx.x * ethreads + etid; i < total; i += (int64_t)gridDim.x * ethreads) yz[i] = 0;
    }
    // factor, cast and store 32 consecutive outputs of row m from n0
    auto store32 = [&](const uint32_t (&r)[32], int64_t m, int64_t n0, float fac, bool zero) {
      constexpr bool kRowScale = !std::is_same<T, TO>::value;
      const float rsc = row_factor<T, TO>(p, m);
      uint32_t packed[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        float v0 = __uint_as_float(r[2 * k]), v1 = __uint_as_float(r[2 * k + 1]);
        if (kRowScale) {
          v0 *= rsc;
          v1 *= rsc;
        }
        if (p.gs) {
          v0 = __fmul_rn(v0, fac);
          v1 = __fmul_rn(v1, fac);
        }
        packed[k] = zero ? 0u : out_bits<TO>(v0) | (out_bits<TO>(v1) << 16);
      }
      TO* dst = y + m * p.N + n0;
      if (n0 + 32 <= p.N && (p.N % 8) == 0) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          d4[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
      } else {
        uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
        for (int k = 0; k < 32 && n0 + k < p.N; ++k) d16[k] = (uint16_t)(packed[k >> 1] >> (16 * (k & 1)));
      }
    };
    // After a wait gives up (the CTA is aborting) a warp keeps walking its
    // units without touching TMEM or memory, so that the epilogue warps still
    // meet at every named barrier.
    bool dead = false;
    Unit un;
    for (int i = 0; sched.next(un); ++i) {
      const Tile tl = tile_of<GATHER, BM>(p, un.tile, seg, pre);
      const int b = i % NBUF;
      if (!dead && !wait_bar_warp(accFull(b), (i / NBUF) & 1, abort_flag, 7, &g_tc_error)) dead = true;
      tc_fence_after();
      const int rr = 128 * hm + 32 * q + lane;  // row within the tile
      const int64_t m = tl.m0 + rr;
      const bool live = rr < tl.rows;
      bool zero = false;
      if (GATHER && live) {
        const int64_t xr = p.lhs ? (int64_t)__ldg(p.lhs + m) : m;
        zero = xr >= p.B;
      }
      const float fac = global_factor(p.gs, tl.e);
      const int64_t n_base = (int64_t)tl.nt * BN;
      const uint32_t tcol = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * MH * BN + hm * BN);
      if (SK && (un.kb0 != 0 || un.kb1 != p.num_kb)) {
        // A piece of a stream-K tile: add it to the tile's sums, count its
        // k-blocks; the piece that completes the count finishes the tile.
        const int slot = un.tile - p.dp_tiles;
        float* wcol = p.ws + (int64_t)slot * (BM * BN) + rr;  // + column * BM
        if (!dead) {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tcol + (uint32_t)(32 * c), r);
            tmem_ld_wait();
            if (!live || n_base + 32 * c >= p.N) continue;
#pragma unroll
            for (int k = 0; k < 32; ++k) atomicAdd(wcol + (int64_t)(32 * c + k) * BM, __uint_as_float(r[k]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(accEmpty(b));  // the accumulator is free again
        }
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"n"(C::EPI_WARPS * 32) : "memory");
        if (etid == 0) {
          const uint32_t add = (uint32_t)(un.kb1 - un.kb0);
          s_fin = dead ? 0 : (atomicAdd(p.ws_cnt + slot, add) + add == (uint32_t)p.num_kb);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(C::EPI_WARPS * 32) : "memory");
        if (s_fin && !dead) {
          __threadfence();
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            const int64_t n0 = n_base + 32 * c;
            if (!live || n0 >= p.N) continue;
            uint32_t r[32];
            float* src = wcol + (int64_t)(32 * c) * BM;
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__ldcg(src + (int64_t)k * BM));
#pragma unroll
            for (int k = 0; k < 32; ++k) __stcg(src + (int64_t)k * BM, 0.f);
            store32(r, m, n0, fac, false);
          }
          if (etid == 0) atomicExch(p.ws_cnt + slot, 0u);
        }
        continue;
      }
      if (dead) continue;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tcol + (uint32_t)(32 * c), r);
        tmem_ld_wait();
        if (!live) continue;
        const int64_t n0 = n_base + 32 * c;
        if (n0 >= p.N) continue;
        store32(r, m, n0, fac, zero);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accEmpty(b));
    }
  } else if (warp >= C::kWarpProd0) {
    if constexpr (kNT)
      producer_role_sk_nt<T, C>(p, sB, bars, abort_flag, sched, smem_u32(samp));
    else
      producer_role_sk<T, C, GATHER>(p, sB, bars, abort_flag, sched, seg, pre);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpAlloc) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
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

// Stream-K sums and counters, one buffer pair per (device, stream), grown on
// demand and zeroed when made (on a private stream, with the thread's capture
// mode relaxed, so that a call captured into a CUDA graph gets them outside
// the capture); every launch leaves them zeroed again.
struct SkWs {
  float* acc = nullptr;
  uint32_t* cnt = nullptr;
  size_t floats = 0, counters = 0;
};
std::mutex g_sk_mu;
std::map<std::pair<int, uintptr_t>, SkWs> g_sk;
std::vector<void*> g_sk_retired;

cudaError_t zero_private(void* ptr, size_t bytes) {
  cudaStream_t z = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&z, cudaStreamNonBlocking);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(ptr, 0, bytes, z);
  const cudaError_t e2 = cudaStreamSynchronize(z);
  cudaStreamDestroy(z);
  return e != cudaSuccess ? e : e2;
}

cudaError_t sk_workspace(int dev, cudaStream_t st, size_t floats, size_t counters, SkWs* out) {
  std::lock_guard<std::mutex> lock(g_sk_mu);
  SkWs& w = g_sk[{dev, reinterpret_cast<uintptr_t>(st)}];
  if (w.floats < floats || w.counters < counters) {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaError_t e = cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) return e;
    const size_t nf = floats > w.floats ? floats : w.floats, nc = counters > w.counters ? counters : w.counters;
    float* acc = nullptr;
    uint32_t* cnt = nullptr;
    e = cudaMalloc(&acc, nf * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&cnt, nc * sizeof(uint32_t));
    if (e == cudaSuccess) e = zero_private(acc, nf * sizeof(float));
    if (e == cudaSuccess) e = zero_private(cnt, nc * sizeof(uint32_t));
    cudaStreamCaptureMode back = mode;
    cudaThreadExchangeStreamCaptureMode(&back);
    if (e != cudaSuccess) {
      cudaFree(acc);
      cudaFree(cnt);
      return e;
    }
    if (w.acc) g_sk_retired.push_back(w.acc);
    if (w.cnt) g_sk_retired.push_back(w.cnt);
    w.acc = acc;
    w.cnt = cnt;
    w.floats = nf;
    w.counters = nc;
  }
  *out = w;
  return cudaSuccess;
}

bool stream_k_on() { return tc_stream_k(); }

// The stream-K split applies to launches of fewer than two waves whose
// partial wave would be at most 60% full. Measured on [21504, 5376] with
// 256x256 tiles: 168 tiles (1.1 waves, M = 512) 121.6 us split against 125.0
// whole; 252 tiles (1.66 waves, M = 768) 154.7 split against 137.3 whole;
// 84 tiles (M = 256) 72.9 against 73.7; far fewer tiles than SMs (the decode
// linears at M <= 128) 1.1 to 2.9x faster split.
bool split_k(int tiles, int sms) {
  return stream_k_on() && tiles % sms != 0 && tiles < 2 * sms && (int64_t)(tiles % sms) * 5 <= (int64_t)sms * 3;
}

// Fewest k-blocks a CTA takes of the stream-K tiles when they are fewer than
// the SMs (smaller pieces cost more to combine than they save).
constexpr int64_t kMinSkBlocks = 8;

template <typename T, typename C, typename TO = T>
cudaError_t launch_cfg(const void* x, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales, const float* gs,
                       int64_t N, void* y, int sms, cudaStream_t st, const float* row_scale = nullptr) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {BK, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      std::is_same<T, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(&map, dt, 2, const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcParams p;
  p.w = w;
  p.scales = scales;
  p.gs = gs;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_m_tiles = (int)((M + C::BM - 1) / C::BM);
  p.num_n_tiles = (int)((N + C::BN - 1) / C::BN);
  p.num_tiles = p.num_m_tiles * p.num_n_tiles;
  p.num_kb = (int)((K + BK - 1) / BK);
  p.lhs = nullptr;
  p.rhs = nullptr;
  p.B = M;
  p.E = 1;
  p.glu_cols = 0;
  p.glu_act = 0;
  p.row_scale = row_scale;
  // Tiles are dealt whole, round robin, unless they make fewer than two
  // waves with a mostly empty partial wave (split_k): then that wave would
  // idle a large share of the SMs, and all tiles are split evenly by
  // k-blocks instead (stream-K). From two waves on, splitting only the last
  // wave cost more than it saved (M = 2048 on [21504, 5376], 4.4 waves: 365
  // us whole-tile, 371 us split).
  const int T_ = p.num_tiles;
  int grid = T_ < sms ? T_ : sms;
  p.dp_tiles = T_;
  p.sk_tiles = 0;
  if (split_k(T_, sms)) {
    if (T_ > sms) {
      p.dp_tiles = 0;
      grid = sms;
    } else {
      p.dp_tiles = 0;
      const int64_t by_blocks = (int64_t)T_ * p.num_kb / kMinSkBlocks;
      grid = (int)(by_blocks < T_ ? T_ : (by_blocks < sms ? by_blocks : sms));
    }
    p.sk_tiles = T_ - p.dp_tiles;
  }
  p.ws = nullptr;
  p.ws_cnt = nullptr;
  if (p.sk_tiles > 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    SkWs ws;
    cudaError_t e = sk_workspace(dev, st, (size_t)p.sk_tiles * C::BM * C::BN, (size_t)p.sk_tiles, &ws);
    if (e != cudaSuccess) return e;
    p.ws = ws.acc;
    p.ws_cnt = ws.cnt;
  }
  auto kern = p.sk_tiles > 0 ? qmm_tc_sk_kernel<T, C, false, true, false, TO> : qmm_tc_kernel<T, C, false, false, false, TO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM, st>>>(map, p);
  return cudaGetLastError();
}

using Tile256x256 = Cfg<2, 256>;
using Tile256x128 = Cfg<2, 128>;
using Tile128x256 = Cfg<1, 256>;

// Fused gate/up with its activation: weight tiles of 128 gate rows and the
// matching 128 up rows (BN = 256), whole tiles round robin.
template <typename T, typename C, typename TO = T>
cudaError_t launch_glu_cfg(const void* x, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                           const float* gs, int64_t cols, int act, void* y, int sms, cudaStream_t st,
                           const float* row_scale = nullptr) {
  static_assert(C::BN == 256, "a GLU tile is 128 gate rows and 128 up rows");
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {BK, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      std::is_same<T, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(&map, dt, 2, const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcParams p;
  p.w = w;
  p.scales = scales;
  p.gs = gs;
  p.y = y;
  p.M = M;
  p.N = 2 * cols;
  p.K = K;
  p.num_m_tiles = (int)((M + C::BM - 1) / C::BM);
  p.num_n_tiles = (int)((cols + 127) / 128);
  p.num_tiles = p.num_m_tiles * p.num_n_tiles;
  p.num_kb = (int)((K + BK - 1) / BK);
  p.lhs = nullptr;
  p.rhs = nullptr;
  p.B = M;
  p.E = 1;
  p.dp_tiles = p.num_tiles;
  p.sk_tiles = 0;
  p.ws = nullptr;
  p.ws_cnt = nullptr;
  p.glu_cols = cols;
  p.glu_act = act;
  p.row_scale = row_scale;
  const int grid = p.num_tiles < sms ? p.num_tiles : sms;
  auto kern = qmm_tc_kernel<T, C, false, true, false, TO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM, st>>>(map, p);
  return cudaGetLastError();
}

// Tile shape. Below two waves of 256x256 tiles (split by k-blocks, or one
// wave and a mostly full second one), 256x256 tiles, whose decoded weight
// tile feeds twice the MMA work, were the fastest or within 4% of it on every
// such shape measured on GB300 (M = 64 .. 768 at K = 5376, M = 2048 at K =
// 21504).
// Otherwise (or with the stream-K option off) the shape is picked by
// modelled time: whole waves of persistent tiles, each tile's cost its area
// over the shape's relative throughput (measured with full waves at M = 8192,
// [21504, 5376]: 256x128 tiles run at 0.81 of 256x256, 128x256 tiles at
// 0.54). The NVFP4_OPT_TC_TILE option overrides either choice.
int pick_tile(int64_t M, int64_t N, int sms) {
  const int forced = option(kOptTcTile);  // 1 256x256, 2 256x128, 3 128x256
  if (forced >= 1 && forced <= 3) return forced - 1;
  // fewer than two waves of 256x256 tiles
  if (stream_k_on() && ((M + 255) / 256) * ((N + 255) / 256) < 2 * sms) return 0;
  const int bm[3] = {256, 256, 128}, bn[3] = {256, 128, 256};
  const double rate[3] = {1.0, 0.81, 0.54};
  int best = 0;
  double best_t = 1e300;
  for (int c = 0; c < 3; ++c) {
    const double tiles = (double)((M + bm[c] - 1) / bm[c]) * (double)((N + bn[c] - 1) / bn[c]);
    const double waves = std::ceil(tiles / sms);
    const double t = waves * bm[c] * bn[c] / rate[c];
    if (t < best_t - 1e-9) {
      best_t = t;
      best = c;
    }
  }
  return best;
}

cudaError_t gather_buffer(int dev, cudaStream_t st, size_t bytes, void** out);

// bf16 activation rows as f16, for the f16 kernels: output row r takes x row
// lhs[r] (row r without lhs; an index >= B gives a zero row), scaled by 2^s,
// the power of two that brings the row's largest finite magnitude into
// [2^14, 2^15), and rounded to f16; rs[r] = 2^-s undoes the scaling on the
// row's sums. A bf16 value keeps 8 significant bits and f16 11 down to
// 2^-14, so every value of at least 2^-29 times the row's largest converts
// exactly; smaller ones round to a multiple of 2^-24 (after scaling), an
// error below 2^-39 of the row's largest value. Infinities and NaNs pass
// through. One warp per row, kv 16-byte units per row.
__device__ __forceinline__ int f16_row_shift(uint32_t mx) {  // mx: largest finite |value| as bf16 bits
  int sh = mx == 0 ? 0 : 141 - (int)(mx >> 7);                 // largest * 2^sh in [2^14, 2^15)
  return sh > 126 ? 126 : sh;                                  // (subnormal maxima)
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float up) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * up, __uint_as_float(w & 0xFFFF0000u) * up);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t finite_abs_max(uint32_t mx, uint32_t w) {
  const uint32_t lo = w & 0x7FFFu, hi = (w >> 16) & 0x7FFFu;
  if (lo < 0x7F80u) mx = lo > mx ? lo : mx;
  if (hi < 0x7F80u) mx = hi > mx ? hi : mx;
  return mx;
}

// kTPR threads per row (a warp, or several warps of a 256-thread CTA); a row
// of up to kTPR * kUnits 16-byte units is read once and kept in registers
// between the maximum and the conversion, longer rows are read twice. The
// launch picks the smallest group that holds the row: a warp per row up to
// 2048 elements (eight rows per CTA), 128 threads up to 6144, 256 threads up
// to 24576; every row of a 2048-row call with K = 5376 is then resident at
// once, and 32768 short rows do not queue behind each other in one CTA.
template <int kTPR, int kUnits, int kMinBlocks>
__global__ void __launch_bounds__(256, kMinBlocks) rows_to_f16_kernel(const uint4* __restrict__ x,
                                                                      const uint32_t* __restrict__ lhs, int64_t B,
                                                                      int64_t R, int kv, uint4* __restrict__ xh,
                                                                      float* __restrict__ rs) {
  constexpr int kGroups = 256 / kTPR, kWarpsPerRow = kTPR / 32;
  __shared__ uint32_t s_max[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, grp = tid / kTPR, gtid = tid % kTPR;
  // every thread of the CTA takes the same number of turns (the barriers)
  for (int64_t base = (int64_t)blockIdx.x * kGroups; base < R; base += (int64_t)gridDim.x * kGroups) {
    const int64_t r = base + grp;
    const bool has = r < R;
    const int64_t src = has ? (lhs ? (int64_t)__ldg(lhs + r) : r) : B;
    const bool live = src < B;  // uniform over the row's group
    const uint4* row = x + (live ? src : 0) * kv;
    const bool in_regs = kv <= kTPR * kUnits;
    uint4 v[kUnits];
    uint32_t mx = 0;
    if (in_regs) {
#pragma unroll
      for (int i = 0; i < kUnits; ++i) {
        const int j = gtid + i * kTPR;
        v[i] = live && j < kv ? __ldg(row + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kUnits; ++i)
        mx = finite_abs_max(finite_abs_max(finite_abs_max(finite_abs_max(mx, v[i].x), v[i].y), v[i].z), v[i].w);
    } else if (live) {
      for (int j = gtid; j < kv; j += kTPR) {
        const uint4 u = __ldg(row + j);
        mx = finite_abs_max(finite_abs_max(finite_abs_max(finite_abs_max(mx, u.x), u.y), u.z), u.w);
      }
    }
    mx = __reduce_max_sync(0xffffffffu, mx);  // a warp never spans two rows
    if constexpr (kWarpsPerRow > 1) {
      if (lane == 0) s_max[warp] = mx;
      __syncthreads();
#pragma unroll
      for (int w = 0; w < kWarpsPerRow; ++w) {
        const uint32_t o = s_max[grp * kWarpsPerRow + w];
        mx = o > mx ? o : mx;
      }
      __syncthreads();  // s_max is rewritten on the next turn
    }
    if (!has) continue;
    const int sh = f16_row_shift(mx);  // 0 for a zero row
    const float up = __uint_as_float((uint32_t)(sh + 127) << 23);
    if (gtid == 0) rs[r] = __uint_as_float((uint32_t)(127 - sh) << 23);
    uint4* out = xh + r * kv;
    if (in_regs) {
#pragma unroll
      for (int i = 0; i < kUnits; ++i) {
        const int j = gtid + i * kTPR;
        if (j < kv)
          out[j] = make_uint4(bf16x2_to_f16x2_scaled(v[i].x, up), bf16x2_to_f16x2_scaled(v[i].y, up),
                              bf16x2_to_f16x2_scaled(v[i].z, up), bf16x2_to_f16x2_scaled(v[i].w, up));
      }
    } else {
      for (int j = gtid; j < kv; j += kTPR) {
        const uint4 u = live ? __ldg(row + j) : make_uint4(0, 0, 0, 0);
        out[j] = make_uint4(bf16x2_to_f16x2_scaled(u.x, up), bf16x2_to_f16x2_scaled(u.y, up),
                            bf16x2_to_f16x2_scaled(u.z, up), bf16x2_to_f16x2_scaled(u.w, up));
      }
    }
  }
}

// The same for rows of any length K, written with kp >= K elements (columns
// past K are +0), for activations that are no TMA source as they are.
__global__ void __launch_bounds__(256) rows_to_f16_pad_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                              int64_t kp, uint16_t* __restrict__ xh,
                                                              float* __restrict__ rs) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < M; r += nwarps) {
    const uint16_t* row = x + r * K;
    uint32_t mx = 0;
    for (int64_t c = lane; c < K; c += 32) mx = finite_abs_max(mx, __ldg(row + c));
    const int sh = f16_row_shift(__reduce_max_sync(0xffffffffu, mx));
    const float up = __uint_as_float((uint32_t)(sh + 127) << 23);
    if (lane == 0) rs[r] = __uint_as_float((uint32_t)(127 - sh) << 23);
    for (int64_t c = lane; c < kp; c += 32) {
      const uint32_t v = c < K ? (uint32_t)__ldg(row + c) : 0u;
      xh[r * kp + c] = (uint16_t)bf16x2_to_f16x2_scaled(v, up);
    }
  }
}

// bf16 activations take the f16 kernels (their weight decode costs about a
// third of the bf16 one: there is no E2M1 -> bf16 conversion): R rows (row r
// from x row lhs[r], or r) are first converted into the stream's scratch
// buffer, rows of kp elements (kp = K when K % 8 == 0), each with a
// power-of-two scale that the kernels undo on its sums.
cudaError_t rows_to_f16(const void* x, int64_t R, int64_t K, const uint32_t* lhs, int64_t B, int sms, cudaStream_t st,
                        const void** xh, const float** rs, int64_t* kp_out = nullptr) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t kp = (K + 7) / 8 * 8;
  const size_t xb = ((size_t)R * (size_t)kp * 2 + 255) / 256 * 256;
  void* buf = nullptr;
  cudaError_t e = gather_buffer(dev, st, xb + (size_t)R * 4, &buf);
  if (e != cudaSuccess) return e;
  float* scale = reinterpret_cast<float*>(static_cast<char*>(buf) + xb);
  const int kv = (int)(K / 8);
  auto grid_for = [&](int64_t rows_per_cta) {
    const int64_t b = (R + rows_per_cta - 1) / rows_per_cta;
    return (unsigned)(b < 16 * sms ? b : 16 * sms);
  };
  if (kp == K && kv <= 32 * 8) {
    rows_to_f16_kernel<32, 8, 3><<<grid_for(8), 256, 0, st>>>(static_cast<const uint4*>(x), lhs, B, R, kv,
                                                             static_cast<uint4*>(buf), scale);
  } else if (kp == K && kv <= 128 * 6) {
    rows_to_f16_kernel<128, 6, 4><<<grid_for(2), 256, 0, st>>>(static_cast<const uint4*>(x), lhs, B, R, kv,
                                                              static_cast<uint4*>(buf), scale);
  } else if (kp == K) {
    rows_to_f16_kernel<256, 12, 3><<<grid_for(1), 256, 0, st>>>(static_cast<const uint4*>(x), lhs, B, R, kv,
                                                               static_cast<uint4*>(buf), scale);
  } else {  // (no row gather with K % 8 != 0: the gather route needs K % 16 == 0)
    const int64_t blocks = (R + 7) / 8;
    rows_to_f16_pad_kernel<<<(unsigned)(blocks < 8 * sms ? blocks : 8 * sms), 256, 0, st>>>(
        static_cast<const uint16_t*>(x), R, K, kp, static_cast<uint16_t*>(buf), scale);
  }
  *xh = buf;
  *rs = scale;
  if (kp_out) *kp_out = kp;
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_tc(const void* x, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales, const float* gs,
                      int64_t N, void* y, cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const float* rs = nullptr;
  if (std::is_same<T, __nv_bfloat16>::value) {
    cudaError_t e = rows_to_f16(x, M, K, nullptr, M, sms, st, &x, &rs);
    if (e != cudaSuccess) return e;
  }
  switch (pick_tile(M, N, sms)) {  // T here is the output type; the kernels decode and multiply in f16
    case 0: return launch_cfg<__half, Tile256x256, T>(x, M, K, w, scales, gs, N, y, sms, st, rs);
    case 1: return launch_cfg<__half, Tile256x128, T>(x, M, K, w, scales, gs, N, y, sms, st, rs);
    default: return launch_cfg<__half, Tile128x256, T>(x, M, K, w, scales, gs, N, y, sms, st, rs);
  }
}

// Activation rows in output-row order for the expert-batched route: xg[r] =
// x[lhs[r]], zeros where lhs[r] >= B; kv 16-byte units per row. One warp per
// row, four loads in flight per lane.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, const uint32_t* __restrict__ lhs,
                                                          int64_t B, int64_t R, int kv, uint4* __restrict__ xg) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < R; r += nwarps) {
    const int64_t src = (int64_t)__ldg(lhs + r);
    uint4* dst = xg + r * kv;
    if (src >= B) {
      for (int j = lane; j < kv; j += 32) dst[j] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* row = x + src * kv;
    for (int j0 = lane; j0 < kv; j0 += 128) {
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = j0 + 32 * q;
        v[q] = j < kv ? __ldg(row + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = j0 + 32 * q;
        if (j < kv) dst[j] = v[q];
      }
    }
  }
}

// Buffer for the gathered activations, one per (device, stream), grown on
// demand and kept until release_gather_workspaces(). Allocated with the
// thread's capture mode relaxed, so a call captured into a CUDA graph gets it
// outside the capture (as the decode route's workspace).
std::mutex g_xg_mu;
std::map<std::pair<int, uintptr_t>, std::pair<void*, size_t>> g_xg;
std::vector<void*> g_xg_retired;

cudaError_t gather_buffer(int dev, cudaStream_t st, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lock(g_xg_mu);
  auto& slot = g_xg[{dev, reinterpret_cast<uintptr_t>(st)}];
  if (slot.second < bytes) {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaError_t e = cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) return e;
    void* ptr = nullptr;
    e = cudaMalloc(&ptr, bytes);
    cudaStreamCaptureMode back = mode;
    cudaThreadExchangeStreamCaptureMode(&back);
    if (e != cudaSuccess) return e;
    if (slot.first) g_xg_retired.push_back(slot.first);
    slot = {ptr, bytes};
  }
  *out = slot.first;
  return cudaSuccess;
}

// Expert-batched GatherQMM, persistent grid of one CTA per SM; the tile count
// is known only on the device. A tile covers up to C::BM rows of one expert's
// segment; a tile whose rows fit one 128-row half computes only that half.
// With activation indices the rows are first gathered into output-row order,
// so that every activation tile is a plain 128-row TMA box (per-row
// tile::gather4 copies, four rows each and 32 per box, left the copy engine,
// not the tensor core, setting the pace).
template <typename T, typename C, typename TO = T>
cudaError_t launch_gather(const void* x, int64_t B, int64_t K, const uint32_t* lhs, const uint32_t* rhs, int64_t R,
                          const uint32_t* w, const uint8_t* scales, const float* gs, int64_t E, int64_t N, void* y,
                          cudaStream_t st) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const void* xa = x;
  int64_t xrows = B;
  const float* rs = nullptr;
  if (!std::is_same<T, TO>::value) {  // bf16 rows, gathered and converted in one pass
    cudaError_t e = rows_to_f16(x, R, K, lhs, B, sms, st, &xa, &rs);
    if (e != cudaSuccess) return e;
    xrows = R;
  } else if (lhs) {
    void* xg = nullptr;
    cudaError_t e = gather_buffer(dev, st, (size_t)R * (size_t)K * 2, &xg);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (R + 7) / 8;
    gather_rows_kernel<<<(unsigned)(blocks < 4 * sms ? blocks : 4 * sms), 256, 0, st>>>(
        static_cast<const uint4*>(x), lhs, B, R, (int)(K / 8), static_cast<uint4*>(xg));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    xa = xg;
    xrows = R;
  }
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)xrows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {BK, 128u};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      std::is_same<T, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(&map, dt, 2, const_cast<void*>(xa), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcParams p;
  p.w = w;
  p.scales = scales;
  p.gs = gs;
  p.y = y;
  p.M = R;
  p.N = N;
  p.K = K;
  p.num_m_tiles = 0;
  p.num_n_tiles = (int)((N + C::BN - 1) / C::BN);
  p.num_tiles = 0;  // counted on the device
  p.num_kb = (int)((K + BK - 1) / BK);
  p.lhs = lhs;  // still read by the epilogue: rows with an index >= B are +0
  p.rhs = rhs;
  p.B = B;
  p.E = (int)E;
  p.glu_cols = 0;
  p.glu_act = 0;
  p.row_scale = rs;
  const size_t smem = C::SMEM + kGatherSmem;
  auto kern = qmm_tc_kernel<T, C, true, false, false, TO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<sms, C::THREADS, smem, st>>>(map, p);
  return cudaGetLastError();
}

// Gather tile: 256 rows (two halves) by default; the NVFP4_OPT_GATHER_TILE
// option selects 256x128 or 128x256 instead.
template <typename T>
cudaError_t launch_gather_t(const void* x, int64_t B, int64_t K, const uint32_t* lhs, const uint32_t* rhs, int64_t R,
                            const uint32_t* w, const uint8_t* scales, const float* gs, int64_t E, int64_t N, void* y,
                            cudaStream_t st) {
  // T is the activation (and output) type; the kernels decode and multiply in f16
  const int t = option(kOptGatherTile);  // 0 or 1 256x256, 2 256x128, 3 128x256
  if (t == 3) return launch_gather<__half, Tile128x256, T>(x, B, K, lhs, rhs, R, w, scales, gs, E, N, y, st);
  if (t == 2) return launch_gather<__half, Tile256x128, T>(x, B, K, lhs, rhs, R, w, scales, gs, E, N, y, st);
  return launch_gather<__half, Tile256x256, T>(x, B, K, lhs, rhs, R, w, scales, gs, E, N, y, st);
}

// Activations whose rows are not a multiple of 16 bytes (K % 8 != 0) cannot
// be a TMA source: they are copied with rows of kp >= K elements, the columns
// past K set to +0.
__global__ void __launch_bounds__(256) pad_cols_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t kp,
                                                       uint16_t* __restrict__ xp) {
  const int64_t n = M * kp;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / kp, c = i - m * kp;
    xp[i] = c < K ? x[m * K + c] : (uint16_t)0;
  }
}

// Non-transposed weights ([K, N/8] words, scales along N): whole tiles dealt
// round robin to a persistent grid; 128-row tiles while M fits one.
template <typename T, typename C, typename TO = T>
cudaError_t launch_nt_cfg(const void* x, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                          const float* gs, int64_t N, void* y, int sms, cudaStream_t st) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const void* xa = x;
  int64_t kx = K;
  const float* rs = nullptr;
  if (!std::is_same<T, TO>::value) {  // bf16 rows: converted (and padded) in one pass
    cudaError_t e = rows_to_f16(x, M, K, nullptr, M, sms, st, &xa, &rs, &kx);
    if (e != cudaSuccess) return e;
  } else if (K % 8) {
    int dev = 0;
    cudaGetDevice(&dev);
    kx = (K + 7) / 8 * 8;
    void* xp = nullptr;
    cudaError_t e = gather_buffer(dev, st, (size_t)M * (size_t)kx * 2, &xp);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (M * kx + 255) / 256;
    pad_cols_kernel<<<(unsigned)(blocks < 4 * sms ? blocks : 4 * sms), 256, 0, st>>>(
        static_cast<const uint16_t*>(x), M, K, kx, static_cast<uint16_t*>(xp));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    xa = xp;
  }
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)kx, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)kx * 2};
  const cuuint32_t box[2] = {BK, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      std::is_same<T, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(&map, dt, 2, const_cast<void*>(xa), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcParams p;
  p.w = w;
  p.scales = scales;
  p.gs = gs;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_m_tiles = (int)((M + C::BM - 1) / C::BM);
  p.num_n_tiles = (int)((N + C::BN - 1) / C::BN);
  p.num_tiles = p.num_m_tiles * p.num_n_tiles;
  p.num_kb = (int)((K + BK - 1) / BK);
  p.lhs = nullptr;
  p.rhs = nullptr;
  p.B = M;
  p.E = 1;
  p.glu_cols = 0;
  p.glu_act = 0;
  p.row_scale = rs;
  // the dense route's rule: below two waves of tiles (and not whole waves)
  // every tile's k-blocks are split evenly over the CTAs
  const int T_ = p.num_tiles;
  int grid = T_ < sms ? T_ : sms;
  p.dp_tiles = T_;
  p.sk_tiles = 0;
  p.ws = nullptr;
  p.ws_cnt = nullptr;
  if (split_k(T_, sms)) {
    p.dp_tiles = 0;
    p.sk_tiles = T_;
    if (T_ > sms) {
      grid = sms;
    } else {
      const int64_t by_blocks = (int64_t)T_ * p.num_kb / kMinSkBlocks;
      grid = (int)(by_blocks < T_ ? T_ : (by_blocks < sms ? by_blocks : sms));
    }
    int dev = 0;
    cudaGetDevice(&dev);
    SkWs ws;
    cudaError_t e = sk_workspace(dev, st, (size_t)p.sk_tiles * C::BM * C::BN, (size_t)p.sk_tiles, &ws);
    if (e != cudaSuccess) return e;
    p.ws = ws.acc;
    p.ws_cnt = ws.cnt;
  }
  auto kern = p.sk_tiles > 0 ? qmm_tc_sk_kernel<T, C, false, true, true, TO> : qmm_tc_kernel<T, C, false, false, true, TO>;
  const size_t smem = C::SMEM + 1024;  // + the producer's scale table
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, smem, st>>>(map, p);
  return cudaGetLastError();
}

}  // namespace

bool gather_tc_supported(int64_t B, int64_t K, int64_t R, int64_t E, int64_t N) {
  // 32-bit activation-row coordinates and row counts; K as for the dense route
  return B > 0 && B < (1ll << 31) && R > 0 && R < (1ll << 31) && E >= 1 && E <= kGatherMaxE && N > 0 && K >= 32 &&
         K % 32 == 0 && K < (1ll << 31) && ((R + 127) / 128 + E) * ((N + 127) / 128) < (1ll << 31);
}

cudaError_t launch_gather_tc(const void* x, int xdt, int64_t B, int64_t K, const uint32_t* lhs, const uint32_t* rhs,
                             int64_t R, const uint32_t* w, const uint8_t* scales, const float* gs, int64_t E, int64_t N,
                             void* y, cudaStream_t st) {
  if (xdt == kBF16) return launch_gather_t<__nv_bfloat16>(x, B, K, lhs, rhs, R, w, scales, gs, E, N, y, st);
  return launch_gather_t<__half>(x, B, K, lhs, rhs, R, w, scales, gs, E, N, y, st);
}

cudaError_t launch_qmm_tc_glu(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                              const float* gs, int64_t cols, int act, void* y, cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (xdt == kBF16) {  // through the f16 kernel (rows_to_f16)
    const float* rs = nullptr;
    cudaError_t e = rows_to_f16(x, M, K, nullptr, M, sms, st, &x, &rs);
    if (e != cudaSuccess) return e;
    return M <= 128
               ? launch_glu_cfg<__half, Tile128x256, __nv_bfloat16>(x, M, K, w, scales, gs, cols, act, y, sms, st, rs)
               : launch_glu_cfg<__half, Tile256x256, __nv_bfloat16>(x, M, K, w, scales, gs, cols, act, y, sms, st, rs);
  }
  return M <= 128 ? launch_glu_cfg<__half, Tile128x256>(x, M, K, w, scales, gs, cols, act, y, sms, st)
                  : launch_glu_cfg<__half, Tile256x256>(x, M, K, w, scales, gs, cols, act, y, sms, st);
}

bool qmm_tc_nt_supported(int64_t M, int64_t N, int64_t K) {
  return M > 0 && N > 0 && N % 16 == 0 && K > 0 && M < (1ll << 31) && K < (1ll << 31) &&
         (M + 127) / 128 * ((N + 255) / 256) < (1ll << 31);
}

cudaError_t launch_qmm_tc_nt(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                             const float* gs, int64_t N, void* y, cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (xdt == kBF16)  // through the f16 kernels (rows_to_f16)
    return M <= 128 ? launch_nt_cfg<__half, Tile128x256, __nv_bfloat16>(x, M, K, w, scales, gs, N, y, sms, st)
                    : launch_nt_cfg<__half, Tile256x256, __nv_bfloat16>(x, M, K, w, scales, gs, N, y, sms, st);
  return M <= 128 ? launch_nt_cfg<__half, Tile128x256>(x, M, K, w, scales, gs, N, y, sms, st)
                  : launch_nt_cfg<__half, Tile256x256>(x, M, K, w, scales, gs, N, y, sms, st);
}

bool tc_stream_k() { return option(kOptTcStreamK) != 0; }

bool qmm_tc_supported(int64_t M, int64_t N, int64_t K) {
  // TMA coordinates are 32-bit; K must keep each 128-bit weight load within
  // one k-block row segment (K % 32 == 0).
  return M > 0 && N > 0 && K >= 32 && K % 32 == 0 && M < (1ll << 31) && K < (1ll << 31) &&
         (M + 127) / 128 * ((N + 127) / 128) < (1ll << 31);
}

cudaError_t launch_qmm_tc(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                          const float* gs, int64_t N, void* y, cudaStream_t st) {
  if (xdt == kBF16) return launch_tc<__nv_bfloat16>(x, M, K, w, scales, gs, N, y, st);
  return launch_tc<__half>(x, M, K, w, scales, gs, N, y, st);
}

void release_gather_workspaces() {
  {
    std::lock_guard<std::mutex> lock(g_xg_mu);
    for (auto& kv : g_xg) cudaFree(kv.second.first);
    g_xg.clear();
    for (void* ptr : g_xg_retired) cudaFree(ptr);
    g_xg_retired.clear();
  }
  std::lock_guard<std::mutex> lock(g_sk_mu);
  for (auto& kv : g_sk) {
    cudaFree(kv.second.acc);
    cudaFree(kv.second.cnt);
  }
  g_sk.clear();
  for (void* ptr : g_sk_retired) cudaFree(ptr);
  g_sk_retired.clear();
}

int read_tc_error() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
  return v;
}

}  // namespace nvfp4
