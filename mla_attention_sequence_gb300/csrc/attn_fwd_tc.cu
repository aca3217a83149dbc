// Causal attention forward on the tensor cores for the LAGA MLA block:
// d_qk = 128 (no-RoPE) + 64 (RoPE), d_v = 128, bf16 operands, fp32 softmax.
//
// One CTA per (128-row query tile, head, batch element); keys stream in
// 128-row tiles. The RoPE-key concat of each head is never materialised:
// S = Q K^T is the sum of the no-RoPE product (K = 128) and the RoPE product
// against the shared k_rope tile (K = 64), accumulated into one TMEM tile.
//
// Warp roles (256 threads):
//   warp 0      lane 0: TMA for Q once, then K tiles
//   warp 1      TMEM allocation; the whole warp runs the MMA issue loop and
//               touches no shared memory in it: it learns that an operand is
//               ready from warp 7 through a named barrier
//   warp 7      the waiter: waits on each mbarrier the next MMA group needs, then
//               meets warp 1 at the named barrier (the AND of their flags
//               carries a timeout)
//   warps 2..5  softmax: one query row per thread (TMEM lane), online max and
//               sum in the log2 domain, P written back over S as bf16 pairs,
//               O rescaled in TMEM when the running max grows, final epilogue
//   warp 6      lane 0: TMA for V tiles
// TMEM columns: three S/P buffers [0,128), [128,256), [256,384); O [384,512).
// With three buffers the score tile S(j+1) is ready before the softmax of tile
// j ends: MMA order S(0) S(1) S(2) PV(0) S(3) PV(1) S(4) ..., S(j+3) reusing the
// buffer that PV(j) has just read. The softmax warps then run back to back and
// the step costs the larger of the MMA time and the softmax time rather than a
// chain of both.
#include "internal.h"
#include "ptx.cuh"

LAGA_TRACE_DEFINE(fwd)

namespace laga {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int BOX = 16384;  // one [128 rows][64 cols] bf16 box
constexpr int Q_BYTES = 3 * BOX;
constexpr int K_BYTES = 3 * BOX;
constexpr int V_BYTES = 2 * BOX;
constexpr int K_STAGES = 2;
constexpr int V_STAGES = 2;
constexpr int NBUF = 3;  // S/P buffers in TMEM
// K/V tiles are prefetched into L2 this many tiles ahead of their TMA load.
constexpr int PREFETCH = 4;
constexpr int SMEM_BYTES = Q_BYTES + K_STAGES * K_BYTES + V_STAGES * V_BYTES + 1024 + 256;
constexpr int NTHREADS = 256;
static_assert(4 * 8192 <= Q_BYTES, "the epilogue stages 4 warps x 8 KB in the Q tile's space");
constexpr int WAITER_WARP = 7;
constexpr int HANDOFF_BAR = 1;  // named barrier of warp 1 and the waiter (64 threads)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 384;
constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 128, false, true);
constexpr float LOG2E = 1.4426950408889634f;
// The running max is only raised (and O rescaled) once it has grown by more
// than this many powers of two; exact, since numerator and denominator share
// the stale max.
constexpr float RESCALE_THRESHOLD = 8.0f;

struct FwdParams {
  int* status;  // device status word (timeouts)
  int Sq, S, n_h, q_offset, causal, skv_pad, n_q_tiles;
  int q_split, q_offset2;  // second query segment (q_split = 0: none)
  float scale_log2;  // softmax scale * log2(e), > 0
  float* lse;
};

// Absolute position of local query row i (a query tile never straddles the
// segments: q_split is a multiple of the tile height).
__device__ __forceinline__ int q_pos(const FwdParams& p, int i) {
  return (p.q_split > 0 && i >= p.q_split) ? p.q_offset2 + (i - p.q_split) : p.q_offset + i;
}

__device__ __forceinline__ int n_kv_tiles(const FwdParams& p, int t) {
  const int last = p.causal ? q_pos(p, min(p.Sq, (t + 1) * BQ) - 1) : p.S - 1;
  return last / BKV + 1;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mR, const __grid_constant__ CUtensorMap mV,
                    const __grid_constant__ CUtensorMap mO, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  LAGA_TRACE_CTA_BEGIN(fwd);
  LAGA_TRACE_POINT(fwd, 30, 0);
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + Q_BYTES;
  uint8_t* sV = sK + K_STAGES * K_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + V_STAGES * V_BYTES);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = q_full + 1;          // [K_STAGES]
  uint64_t* k_empty = k_full + K_STAGES;  // [K_STAGES]
  uint64_t* v_full = k_empty + K_STAGES;  // [V_STAGES]
  uint64_t* v_empty = v_full + V_STAGES;  // [V_STAGES]
  uint64_t* s_full = v_empty + V_STAGES;  // [NBUF]
  uint64_t* p_full = s_full + NBUF;       // [NBUF]
  uint64_t* pv_done = p_full + NBUF;      // [NBUF] PV(j) -> pv_done[j % NBUF]
  uint64_t* drain = pv_done + NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  static_assert((2 + 2 * K_STAGES + 2 * V_STAGES + 3 * NBUF) * 8 + 8 <= 256, "barrier area");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heaviest query tiles (most key tiles) first.
  const int t = p.n_q_tiles - 1 - static_cast<int>(blockIdx.x);
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int n_kv = n_kv_tiles(p, t);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < K_STAGES; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < V_STAGES; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mR);
      mbar_arrive_expect_tx(q_full, Q_BYTES);
      tma_load_3d(sQ, &mQ, q_full, h * 192, t * BQ, b);
      tma_load_3d(sQ + BOX, &mQ, q_full, h * 192 + 64, t * BQ, b);
      tma_load_3d(sQ + 2 * BOX, &mQ, q_full, h * 192 + 128, t * BQ, b);
      int j = 0;
      for (; j < n_kv; ++j) {
        const int s = j % K_STAGES;
        if (!mbar_wait_or_abort(&k_empty[s], ((j / K_STAGES) & 1) ^ 1, abort_flag, 11)) break;
        LAGA_TRACE_POINT(fwd, 20, j);
        uint8_t* dst = sK + s * K_BYTES;
        mbar_arrive_expect_tx(&k_full[s], K_BYTES);
        const int row = b * p.skv_pad + j * BKV;
        tma_load_2d(dst, &mK, &k_full[s], h * 128, row);
        tma_load_2d(dst + BOX, &mK, &k_full[s], h * 128 + 64, row);
        tma_load_3d(dst + 2 * BOX, &mR, &k_full[s], 0, j * BKV, b);
        if (j + PREFETCH < n_kv) {
          tma_prefetch_2d(&mK, h * 128, row + PREFETCH * BKV);
          tma_prefetch_2d(&mK, h * 128 + 64, row + PREFETCH * BKV);
        }
      }
      if (j < n_kv) {  // aborted: let issued copies land
        mbar_drain(q_full, 0);
        for (int i = j - K_STAGES < 0 ? 0 : j - K_STAGES; i < j; ++i)
          mbar_drain(&k_full[i % K_STAGES], (i / K_STAGES) & 1);
      }
    }
  } else if (warp == 6) {
    if (lane == 0) {
      tma_prefetch_desc(&mV);
      int j = 0;
      for (; j < n_kv; ++j) {
        const int s = j % V_STAGES;
        LAGA_TRACE_POINT(fwd, 24, j);
        if (!mbar_wait_or_abort(&v_empty[s], ((j / V_STAGES) & 1) ^ 1, abort_flag, 12)) break;
        LAGA_TRACE_POINT(fwd, 21, j);
        uint8_t* dst = sV + s * V_BYTES;
        mbar_arrive_expect_tx(&v_full[s], V_BYTES);
        const int row = b * p.skv_pad + j * BKV;
        tma_load_2d(dst, &mV, &v_full[s], h * 128, row);
        tma_load_2d(dst + BOX, &mV, &v_full[s], h * 128 + 64, row);
        if (j + PREFETCH < n_kv) {
          tma_prefetch_2d(&mV, h * 128, row + PREFETCH * BKV);
          tma_prefetch_2d(&mV, h * 128 + 64, row + PREFETCH * BKV);
        }
      }
      if (j < n_kv)
        for (int i = j - V_STAGES < 0 ? 0 : j - V_STAGES; i < j; ++i)
          mbar_drain(&v_full[i % V_STAGES], (i / V_STAGES) & 1);
    }
  } else if (warp == WAITER_WARP) {
    // The waiter walks the MMA warp's waits in the same order: q_full, then per
    // iteration j p_full(j) and v_full(j) (j >= 0, one hand-off) and k_full(j+3)
    // (j + 3 < n). A failed wait (timeout or abort) is ANDed in at the named
    // barrier, and both warps leave their loops at the same hand-off.
    if (bar_and(HANDOFF_BAR, 64, warp_wait_or_abort(q_full, 0, abort_flag, 13))) {
      for (int j = -NBUF; j < n_kv; ++j) {
        const int jn = j + NBUF;
        if (j >= 0) {
          const bool w = warp_wait_or_abort(&p_full[j % NBUF], (j / NBUF) & 1, abort_flag, 14) &&
                         warp_wait_or_abort(&v_full[j % V_STAGES], (j / V_STAGES) & 1, abort_flag, 15);
          if (!bar_and(HANDOFF_BAR, 64, w)) break;
        }
        if (jn < n_kv &&
            !bar_and(HANDOFF_BAR, 64, warp_wait_or_abort(&k_full[jn % K_STAGES], (jn / K_STAGES) & 1, abort_flag, 16)))
          break;
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop; an elected lane issues each block of
    // four MMAs. One loop issues everything (code run once per CTA falls out of the
    // instruction cache between CTAs and then issues several times slower).
    // Iteration j: PV(j) (j >= 0), then S(j+3) (j+3 < n). Readiness of every
    // operand comes from the waiter through the named barrier.
    auto ready = [&]() -> bool {
      const bool r = bar_and(HANDOFF_BAR, 64, true);
      tc_fence_after();
      return r;
    };
    bool ok = ready();  // Q
    bool issued = false;
    const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
#ifdef LAGA_TRACE
    // trace build only: cycles spent at each hand-off
    long long st_cyc[3] = {0, 0, 0};
    const long long st_t0 = clock64();
#endif
    for (int j = -NBUF; j < n_kv && ok; ++j) {
      const int jn = j + NBUF;
      if (j >= 0) {
        const int vs = j % V_STAGES;
#ifdef LAGA_TRACE
        const long long w0 = clock64();
#endif
        if (!ready()) {  // P(j) and V(j)
          ok = false;
          break;
        }
#ifdef LAGA_TRACE
        st_cyc[0] += clock64() - w0;
#endif
        if (lane == 0) LAGA_TRACE_POINT(fwd, 3, j);
        const uint64_t v_desc = sdesc_sw128(smem_u32(sV + vs * V_BYTES), BOX, 1024);
        const uint32_t p_tmem = tmem + (j % NBUF) * 128;
#pragma unroll
        for (int g = 0; g < BKV / 64; ++g) {  // keys [64g, 64g + 64): four K16 steps
          const int kk = 4 * g;
          mma4_ts_warp(tmem + COL_O, p_tmem + kk * 8, p_tmem + kk * 8 + 8, p_tmem + kk * 8 + 16, p_tmem + kk * 8 + 24,
                       v_desc + ((kk * 2048) >> 4), v_desc + (((kk + 1) * 2048) >> 4),
                       v_desc + (((kk + 2) * 2048) >> 4), v_desc + (((kk + 3) * 2048) >> 4), IDESC_PV,
                       (j > 0 || g > 0) ? 1u : 0u);
        }
        mma_commit_warp(&pv_done[j % NBUF]);
        mma_commit_warp(&v_empty[vs]);
        if (lane == 0) LAGA_TRACE_POINT(fwd, 5, j);
      }
      if (jn < n_kv) {
        const int ks = jn % K_STAGES;
#ifdef LAGA_TRACE
        const long long w1 = clock64();
#endif
        if (!ready()) {  // K(j+3)
          ok = false;
          break;
        }
#ifdef LAGA_TRACE
        st_cyc[2] += clock64() - w1;
#endif
        if (lane == 0) LAGA_TRACE_POINT(fwd, 1, jn);
        const uint64_t k_desc = sdesc_sw128(smem_u32(sK + ks * K_BYTES), 16, 1024);
#pragma unroll
        for (int c = 0; c < 3; ++c) {  // head dims [64c, 64c + 64): four K16 steps in box c
          const uint32_t o = (c * BOX) >> 4;
          mma4_ss_warp(tmem + (jn % NBUF) * 128, q_desc + o, q_desc + o + 2, q_desc + o + 4, q_desc + o + 6,
                       k_desc + o, k_desc + o + 2, k_desc + o + 4, k_desc + o + 6, IDESC_S, c > 0 ? 1u : 0u);
        }
        issued = true;
        mma_commit_warp(&s_full[jn % NBUF]);
        mma_commit_warp(&k_empty[ks]);
        if (lane == 0) LAGA_TRACE_POINT(fwd, 2, jn);
      }
    }
#ifdef LAGA_TRACE
    if (lane == 0) {
      for (int k = 0; k < 3; ++k) {
        LAGA_TRACE_STAT(fwd, k, 0);
        LAGA_TRACE_STAT(fwd, 3 + k, st_cyc[k]);
      }
      LAGA_TRACE_STAT(fwd, 6, clock64() - st_t0);
      LAGA_TRACE_STAT(fwd, 7, n_kv);
    }
#endif
    if (!ok && issued) {
      mma_commit_warp(drain);
      if (lane == 0) mbar_drain(drain, 0);
      __syncwarp();
    }
  } else {
    // ---------------- softmax warpgroup: thread owns query row r of the tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int q_row = t * BQ + r;  // local query index
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int limit = p.causal ? q_pos(p, q_row) : p.S - 1;  // last visible key
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;  // running max of the scaled (log2-domain) scores
    float l_run = 0.f;
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
      const bool all = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      __syncwarp();  // order lane 0's acquire before the other lanes' reads
      return all;
    };
    for (int j = 0; j < n_kv && ok; ++j) {
      const int buf = j % NBUF;
      // S(j) is issued after PV(j-3), so its completion also means P(j-3) in this
      // buffer has been read.
      if (!warp_wait(&s_full[buf], (j / NBUF) & 1, 18)) {
        ok = false;
        break;
      }
      if (lane == 0) LAGA_TRACE_POINT(fwd, 10, j);
      tc_fence_after();
      const uint32_t s_addr = tmem + buf * 128 + lane_off;
      uint32_t x[128];  // raw fp32 scores of this row
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32 * c));
      tmem_wait_ld();
      const int kv0 = j * BKV;
      if (kv0 + BKV - 1 > limit) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (kv0 + i > limit) x[i] = 0xff800000u;  // -inf
      }
      if (lane == 0) LAGA_TRACE_POINT(fwd, 11, j);
      // max of the raw scores (the scale is positive), four independent chains
      float m4[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) m4[a] = __uint_as_float(x[a]);
#pragma unroll
      for (int i = 4; i < 128; i += 8) {
#pragma unroll
        for (int a = 0; a < 4; ++a)
          m4[a] = max3f(m4[a], __uint_as_float(x[i + 2 * a]), __uint_as_float(x[i + 2 * a + 1]));
      }
      const float mt = max3f(fmaxf(m4[0], m4[1]), m4[2], m4[3]) * sl2;
      float m_use = m_run;
      float alpha = 1.f;
      bool rescale = false;
      if (m_run == -INFINITY) {
        m_use = mt;
      } else if (mt > m_run + RESCALE_THRESHOLD) {
        m_use = mt;
        alpha = ex2_approx(m_run - mt);
        rescale = true;
      }
      // rows with nothing visible yet keep p = 0
      const float neg_m = m_use == -INFINITY ? 0.f : -m_use;
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(x[2 * i]), sl2, neg_m));
        const float p1 = ex2_approx(fmaf(__uint_as_float(x[2 * i + 1]), sl2, neg_m));
        sum2[i & 1] = add_f32x2(sum2[i & 1], make_float2(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + ((sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y));
      m_run = m_use;
      if (lane == 0) LAGA_TRACE_POINT(fwd, 12, j);
      tmem_st32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(pk));
      tmem_st32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      if (__any_sync(0xffffffffu, rescale)) {
        // O may only be touched once PV(j-1) has landed.
        if (j >= 1 && !warp_wait(&pv_done[(j - 1) % NBUF], ((j - 1) / NBUF) & 1, 17)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t o_addr = tmem + COL_O + lane_off;
        uint32_t u[32];
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(o_addr + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(o_addr + c * 32, u);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[buf]);
      if (lane == 0) LAGA_TRACE_POINT(fwd, 13, j);
    }
    if (ok && warp_wait(&pv_done[(n_kv - 1) % NBUF], ((n_kv - 1) / NBUF) & 1, 19)) {
      LAGA_TRACE_POINT(fwd, 29, 0);
      tc_fence_after();
      // Epilogue: O / l as bf16 through shared memory and tensor-map stores, which
      // the TMA unit carries out while the CTA ends (row-per-thread global stores
      // touch 32 lines per instruction and keep the warp busy until they have left
      // the SM). Every MMA has finished, so the Q tile's space is free: each warp
      // stages its 32 rows as two [32 rows][128 B] boxes (128-byte swizzle, the
      // 16-byte chunk k of row r at r * 128 + ((k ^ (r & 7)) << 4)); rows past Sq
      // are clipped by the map.
      const uint32_t o_addr = tmem + COL_O + lane_off;
      const float inv = 1.f / l_run;
      uint8_t* stage = sQ + quarter * 8192;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(o_addr + c * 32, u);
        tmem_wait_ld();
        uint8_t* box = stage + (c >> 1) * 4096 + lane * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(u[8 * v + 0]) * inv, __uint_as_float(u[8 * v + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(u[8 * v + 2]) * inv, __uint_as_float(u[8 * v + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(u[8 * v + 4]) * inv, __uint_as_float(u[8 * v + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(u[8 * v + 6]) * inv, __uint_as_float(u[8 * v + 7]) * inv);
          const uint32_t k = static_cast<uint32_t>((c & 1) * 4 + v);
          *reinterpret_cast<uint4*>(box + ((k ^ (lane & 7u)) << 4)) = w;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&mO, stage, h * 128, t * BQ + quarter * 32, b);
        tma_store_3d(&mO, stage + 4096, h * 128 + 64, t * BQ + quarter * 32, b);
        bulk_commit_group();
        bulk_wait_read_all();  // shared memory must not go away under a store
      }
      __syncwarp();
      if (q_row < p.Sq)
        p.lse[(static_cast<long long>(b) * p.n_h + h) * p.Sq + q_row] =
            (m_run + __log2f(l_run)) * 0.6931471805599453f;
    }
  }

  LAGA_TRACE_POINT(fwd, 28, 0);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) publish_abort(abort_flag, p.status);
  LAGA_TRACE_POINT(fwd, 31, 0);
  LAGA_TRACE_CTA_END(fwd);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

// The [rows][64] boxes of the operands: 3D q map over [B][Sq][n_h*192], 2D maps
// over the [B*skv_pad][n_h*128] K/V workspace, 3D k_rope map over [B][S][64].
LaunchResult tc_attn_fwd(const Dims& d, const bf16* q, const bf16* k_ws, const bf16* v_ws, const bf16* k_rope,
                         bf16* out, float* lse, cudaStream_t st) {
  LaunchResult r;
  CUtensorMap mQ, mK, mR, mV;
  {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 192;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    const uint32_t box[3] = {64, 128, 1};
    r.cu = make_tmap(&mQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t kv_inner = static_cast<uint64_t>(d.n_h) * 128;
  const uint64_t kv_rows = static_cast<uint64_t>(d.B) * d.skv_pad;
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[2] = {kv_inner, kv_rows};
    const uint64_t strides[1] = {kv_inner * 2};
    const uint32_t box[2] = {64, 128};
    r.cu = make_tmap(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k_ws, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r.cu == CUDA_SUCCESS)
      r.cu = make_tmap(&mV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v_ws, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(d.S), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(d.S) * 128};
    const uint32_t box[3] = {64, 128, 1};
    r.cu = make_tmap(&mR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_rope, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  CUtensorMap mO;  // the output's [32 rows][64] boxes, 3D over [B][Sq][n_h*128]: rows past Sq clip
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 128;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    const uint32_t box[3] = {64, 32, 1};
    r.cu = make_tmap(&mO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps attention forward";
    return r;
  }
  FwdParams p{};
  p.Sq = d.Sq;
  p.S = d.S;
  p.n_h = d.n_h;
  p.q_offset = d.q_offset;
  p.q_split = d.q_split;
  p.q_offset2 = d.q_offset2;
  p.causal = d.causal ? 1 : 0;
  p.skv_pad = d.skv_pad;
  p.n_q_tiles = (d.Sq + BQ - 1) / BQ;
  p.scale_log2 = d.scale * LOG2E;
  p.lse = lse;
  p.status = device_status_ptr();
  r.err = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(attn_fwd)";
    return r;
  }
  attn_fwd_kernel<<<dim3(p.n_q_tiles, d.n_h, d.B), NTHREADS, SMEM_BYTES, st>>>(mQ, mK, mR, mV, mO, p);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "attn_fwd_kernel launch";
  return r;
}

}  // namespace laga
