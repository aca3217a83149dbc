// Attention backward, query side: dq on the tensor cores (d_qk = 128 + 64,
// d_v = 128, bf16 operands, fp32 accumulation).
//
// One CTA per (128-row query tile, head, batch element); it walks the 128-row
// key tiles the tile can see and keeps the whole dq tile (192 head dims) in
// TMEM, so every dq element is written once, with no accumulation in memory:
//   S  = Q K^T          P  = exp(S * scale - lse)      (lse from the forward)
//   dP = dO V^T         dS = P o (dP - D)
//   dq += dS K          (scale applied once at the end)
// The RoPE-key concat is folded in as in the forward: S = Q_nope K_nope^T +
// Q_rope k_rope^T, and dq's last 64 columns come from the k_rope tile.
//
// TMEM columns: two step buffers [0,128) and [128,256), dq [256,448), dO
// [448,512). Step j uses buffer j % 2 for all three of its tiles in turn: S(j),
// which the softmax warps copy to registers and release at once; then dP(j);
// then dS(j), packed as bf16 over the dP(j) columns each warpgroup has read,
// from where dq(j) reads it. MMA order S(0) S(1)? dP(0) | dq(j) dP(j+1) S(j+2) |
// ...: dP(j+1) needs only S(j+1) released, not dq(j) done, so the loop-carried
// chain is the tensor work itself (dq 768 + dP 512 + S 768 cycles per 128-key
// step) with the softmax beside it. Measured on GB300 with one S and one dP/dS
// buffer (dP(j+1) after dq(j)): 2425 cycles per step, the softmax's dS half and
// dq(j) + dP(j+1) in one chain.
//
// Warp roles (352 threads):
//   warp 0      lane 0: TMA for Q once, then key tiles
//   warp 1      TMEM allocation; the whole warp runs the MMA issue loop
//   warps 2..9  two warpgroups; each thread owns one query row (TMEM lane) and
//               half of the tile's 128 key columns: P, dS, and half the epilogue
//   warp 10     lane 0: TMA for value tiles
#include "internal.h"
#include "ptx.cuh"

LAGA_TRACE_DEFINE(dq)

namespace laga {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
// K(j) is read by S(j) and, much later, by dq(j); V(j) only by dP(j). Three
// key stages and one value stage fit next to Q.
constexpr int K_STAGES = 3;
constexpr int V_STAGES = 1;
constexpr int BOX = 16384;  // [128 rows][64] bf16
constexpr int Q_BYTES = 3 * BOX;
constexpr int K_BYTES = 3 * BOX;
constexpr int V_BYTES = 2 * BOX;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + Q_BYTES;
static_assert(8 * 6144 <= Q_BYTES, "the epilogue stages 8 warps x 6 KB in the Q tile's space");
constexpr int OFF_V = OFF_K + K_STAGES * K_BYTES;
constexpr int OFF_BARS = OFF_V + V_STAGES * V_BYTES;
constexpr int SMEM_BYTES = OFF_BARS + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_DQ = 256, COL_DO = 448;
// the TMEM buffer of step j (S(j), then dP(j), then dS(j))
__device__ __forceinline__ uint32_t step_buf(int j) { return static_cast<uint32_t>(j & 1) * 128u; }
constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_DQ = idesc_bf16(128, 192, false, true);
constexpr int NTHREADS = 352;
constexpr uint32_t SOFTMAX_WARPS = 8;

struct Params {
  int* status;
  int Sq, S, n_h, q_offset, causal, skv_pad, sq_pad, n_q_tiles;
  int q_split, q_offset2;  // second query segment (q_split = 0: none)
  float scale, scale_log2;
  const float* lse2;
  const float* delta;
  const bf16* dout;  // [B][Sq][n_h][128]
};

// TMEM column of packed bf16 chunk k (16 keys) of dS(j): warpgroup g packs its
// 64 keys into the first 32 columns of its own 64 dP columns, so it never
// overwrites dP values the other warpgroup has not read yet.
__device__ __forceinline__ uint32_t packed_col(int k) { return 8u * (k & 3) + 64u * (k >> 2); }

// Absolute position of local query row i (a query tile never straddles the
// segments: q_split is a multiple of the tile height).
__device__ __forceinline__ int q_pos(const Params& p, int i) {
  return (p.q_split > 0 && i >= p.q_split) ? p.q_offset2 + (i - p.q_split) : p.q_offset + i;
}

__device__ __forceinline__ int n_kv_tiles(const Params& p, int t) {
  const int last = p.causal ? q_pos(p, min(p.Sq, (t + 1) * BQ) - 1) : p.S - 1;
  return last / BKV + 1;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                       const __grid_constant__ CUtensorMap mR, const __grid_constant__ CUtensorMap mV,
                       const __grid_constant__ CUtensorMap mdQ, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  LAGA_TRACE_CTA_BEGIN(dq);
  LAGA_TRACE_POINT(dq, 30, 0);
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [K_STAGES]
  uint64_t* k_empty = bars + 4;  // [K_STAGES]
  uint64_t* v_full = bars + 7;   // [V_STAGES]
  uint64_t* v_empty = bars + 8;  // [V_STAGES]
  uint64_t* s_full = bars + 9;   // S(j) in TMEM
  uint64_t* s_free = bars + 10;  // S(j) copied out by every softmax warp: dP(j) may overwrite it
  uint64_t* dp_full = bars + 11; // dP(j) in TMEM
  uint64_t* ds_full = bars + 12; // dS(j) packed over dP(j)
  uint64_t* dq_done = bars + 13;
  uint64_t* drain = bars + 14;
  uint64_t* do_tmem = bars + 15;  // dO written into TMEM by the query-row warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = p.n_q_tiles - 1 - static_cast<int>(blockIdx.x);  // heaviest tiles first
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
    mbar_init(s_full, 1);
    mbar_init(s_free, SOFTMAX_WARPS);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, SOFTMAX_WARPS);
    mbar_init(dq_done, 1);
    mbar_init(drain, 1);
    mbar_init(do_tmem, SOFTMAX_WARPS);
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
      const int q0 = t * BQ;
      tma_load_3d(smem + OFF_Q, &mQ, q_full, h * 192, q0, b);
      tma_load_3d(smem + OFF_Q + BOX, &mQ, q_full, h * 192 + 64, q0, b);
      tma_load_3d(smem + OFF_Q + 2 * BOX, &mQ, q_full, h * 192 + 128, q0, b);
      int j = 0;
      for (; j < n_kv; ++j) {
        const int s = j % K_STAGES;
        if (!mbar_wait_or_abort(&k_empty[s], ((j / K_STAGES) & 1) ^ 1, abort_flag, 71)) break;
        uint8_t* dst = smem + OFF_K + s * K_BYTES;
        mbar_arrive_expect_tx(&k_full[s], K_BYTES);
        const int row = b * p.skv_pad + j * BKV;
        tma_load_2d(dst, &mK, &k_full[s], h * 128, row);
        tma_load_2d(dst + BOX, &mK, &k_full[s], h * 128 + 64, row);
        tma_load_3d(dst + 2 * BOX, &mR, &k_full[s], 0, j * BKV, b);
      }
      if (j < n_kv) {
        mbar_drain(q_full, 0);
        for (int i = j - K_STAGES < 0 ? 0 : j - K_STAGES; i < j; ++i)
          mbar_drain(&k_full[i % K_STAGES], (i / K_STAGES) & 1);
      }
    }
  } else if (warp == 10) {
    if (lane == 0) {
      tma_prefetch_desc(&mV);
      int j = 0;
      for (; j < n_kv; ++j) {
        const int s = j % V_STAGES;
        if (!mbar_wait_or_abort(&v_empty[s], ((j / V_STAGES) & 1) ^ 1, abort_flag, 72)) break;
        uint8_t* dst = smem + OFF_V + s * V_BYTES;
        mbar_arrive_expect_tx(&v_full[s], V_BYTES);
        const int row = b * p.skv_pad + j * BKV;
        tma_load_2d(dst, &mV, &v_full[s], h * 128, row);
        tma_load_2d(dst + BOX, &mV, &v_full[s], h * 128 + 64, row);
      }
      if (j < n_kv)
        for (int i = j - V_STAGES < 0 ? 0 : j - V_STAGES; i < j; ++i)
          mbar_drain(&v_full[i % V_STAGES], (i / V_STAGES) & 1);
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop; an elected lane issues. One loop issues
    // everything (code run once per CTA falls out of the instruction cache between
    // CTAs and then issues several times slower). Iteration j: dq(j) once dS(j) is
    // in; dP(j+1) once S(j+1) is released; S(j+2) into the buffer dq(j) has just
    // read. Each barrier is tested (without blocking) inside the MMA group that
    // precedes its use, before that group's last block of four, and consumed as a
    // token after the group.
    bool ok = warp_wait_or_abort(q_full, 0, abort_flag, 73) && warp_wait_or_abort(do_tmem, 0, abort_flag, 77);
    bool issued = false;
    tc_fence_after();
    const uint64_t q_desc = sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
    // `tests` runs before the group's last block
    auto issue_s = [&](int j, auto&& tests) {  // S(j) = Q K_j^T
      const uint64_t k_desc = sdesc_sw128(smem_u32(smem + OFF_K + (j % K_STAGES) * K_BYTES), 16, 1024);
#pragma unroll
      for (int c = 0; c < 3; ++c) {  // head dims [64c, 64c + 64): four K16 steps in box c (one elect each)
        if (c == 2) tests();
        const uint32_t o = (c * BOX) >> 4;
        mma4_ss_warp(tmem + step_buf(j), q_desc + o, q_desc + o + 2, q_desc + o + 4, q_desc + o + 6, k_desc + o,
                     k_desc + o + 2, k_desc + o + 4, k_desc + o + 6, IDESC_S, c > 0 ? 1u : 0u);
      }
      mma_commit_warp(s_full);
    };
    auto issue_dp = [&](int j, auto&& tests) {  // dP(j) = dO V_j^T, over S(j)'s columns
      const int s = j % V_STAGES;
      const uint64_t v_desc = sdesc_sw128(smem_u32(smem + OFF_V + s * V_BYTES), 16, 1024);
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // head dims [64c, 64c + 64): dO columns [32c, 32c + 32)
        if (c == 1) tests();
        const uint32_t a = tmem + COL_DO + 32 * c;
        const uint64_t v = v_desc + ((c * BOX) >> 4);
        mma4_ts_warp(tmem + step_buf(j), a, a + 8, a + 16, a + 24, v, v + 2, v + 4, v + 6, IDESC_S,
                     c > 0 ? 1u : 0u);
      }
      mma_commit_warp(dp_full);
      mma_commit_warp(&v_empty[s]);
    };
    uint32_t tk = 0, tv = 0, tf = 0, td = 0;
    for (int j = -2; j < n_kv && ok; ++j) {
      const int j1 = j + 1, j2 = j + 2;
      if (j >= 0) {  // dq(j) += dS(j) K_j : A = dS (TMEM, packed bf16), B = key tile MN-major (N = 192)
        if (!warp_wait_token(ds_full, j & 1, td, abort_flag, 76)) { ok = false; break; }
        tc_fence_after();
        const int s = j % K_STAGES;
        const uint64_t k_mn = sdesc_sw128(smem_u32(smem + OFF_K + s * K_BYTES), BOX, 1024);
        const uint32_t ds = tmem + step_buf(j);
#pragma unroll
        for (int g = 0; g < BKV / 64; ++g) {  // keys [64g, 64g + 64)
          if (g == BKV / 64 - 1 && j1 < n_kv) {
            tf = mbar_test(s_free, j1 & 1);
            tv = mbar_test(&v_full[j1 % V_STAGES], (j1 / V_STAGES) & 1);
          }
          const int k = 4 * g;
          mma4_ts_warp(tmem + COL_DQ, ds + packed_col(k), ds + packed_col(k + 1), ds + packed_col(k + 2),
                       ds + packed_col(k + 3), k_mn + ((k * 2048) >> 4), k_mn + (((k + 1) * 2048) >> 4),
                       k_mn + (((k + 2) * 2048) >> 4), k_mn + (((k + 3) * 2048) >> 4), IDESC_DQ,
                       (j > 0 || g > 0) ? 1u : 0u);
        }
        mma_commit_warp(&k_empty[s]);
      }
      if (j1 >= 0 && j1 < n_kv) {  // dP(j+1): S(j+1) released, V(j+1) in
        if (!warp_wait_token(s_free, j1 & 1, tf, abort_flag, 78)) { ok = false; break; }
        if (!warp_wait_token(&v_full[j1 % V_STAGES], (j1 / V_STAGES) & 1, tv, abort_flag, 75)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_dp(j1, [&]() {
          if (j2 < n_kv) tk = mbar_test(&k_full[j2 % K_STAGES], (j2 / K_STAGES) & 1);
        });
        issued = true;
      }
      if (j2 < n_kv) {  // S(j+2): K(j+2) in; its buffer was last read by dq(j), issued above
        if (!warp_wait_token(&k_full[j2 % K_STAGES], (j2 / K_STAGES) & 1, tk, abort_flag, 74)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(j2, [&]() {
          if (j1 >= 0 && j1 < n_kv) td = mbar_test(ds_full, j1 & 1);
        });
        issued = true;
      } else if (j1 >= 0 && j1 < n_kv) {
        td = mbar_test(ds_full, j1 & 1);
      }
    }
    if (ok) {
      mma_commit_warp(dq_done);
    } else if (issued) {
      mma_commit_warp(drain);
      if (lane == 0) mbar_drain(drain, 0);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------ query-row warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // warpgroup: key columns [64*half, 64*half + 64)
    const int r = quarter * 32 + lane;
    const int q_row = t * BQ + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int limit = p.causal ? q_pos(p, q_row) : p.S - 1;  // last visible key
    const long long roff = (static_cast<long long>(b) * p.n_h + h) * p.sq_pad + q_row;
    const float lse2 = p.lse2[roff];  // +inf on padded rows: P = 0 there
    const float Drow = p.delta[roff];
    const float sl2 = p.scale_log2;
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
      const bool all = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      __syncwarp();  // order lane 0's acquire before the other lanes' reads
      return all;
    };
    // dO row r -> TMEM lane r as packed bf16 pairs (the A-operand layout of a
    // TS-MMA); warpgroup `half` copies head dims [64*half, 64*half + 64).
    {
      const bool valid = q_row < p.Sq;
      const uint4* drow = reinterpret_cast<const uint4*>(
          p.dout + ((static_cast<long long>(b) * p.Sq + (valid ? q_row : 0)) * p.n_h + h) * 128 + 64 * half);
      uint32_t w[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = valid ? __ldg(drow + k) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * k + 0] = v.x;
        w[4 * k + 1] = v.y;
        w[4 * k + 2] = v.z;
        w[4 * k + 3] = v.w;
      }
      tmem_st32(tmem + COL_DO + lane_off + 32 * half, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(do_tmem);
    }
    for (int j = 0; j < n_kv && ok; ++j) {
      const uint32_t ph = j & 1;
      if (!warp_wait(s_full, ph, 81)) { ok = false; break; }
      if (lane == 0) LAGA_TRACE_POINT(dq, 10, j);
      tc_fence_after();
      uint32_t x[64];
      const uint32_t buf = tmem + step_buf(j) + lane_off + 64 * half;
      tmem_ld32(buf, *reinterpret_cast<uint32_t(*)[32]>(x));
      tmem_ld32(buf + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);  // dP(j) may now overwrite S(j)
      const int kv_first = j * BKV + 64 * half;  // this thread's first key column
      float pr[64];
      if (kv_first + 63 <= limit) {  // every key of the half-tile visible
#pragma unroll
        for (int k = 0; k < 64; ++k) pr[k] = ex2_approx(fmaf(__uint_as_float(x[k]), sl2, -lse2));
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          pr[k] = kv_first + k <= limit ? ex2_approx(fmaf(__uint_as_float(x[k]), sl2, -lse2)) : 0.f;
      }
      if (!warp_wait(dp_full, ph, 83)) { ok = false; break; }
      tc_fence_after();
      tmem_ld32(buf, *reinterpret_cast<uint32_t(*)[32]>(x));
      tmem_ld32(buf + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
      tmem_wait_ld();
      uint32_t w[32];
#pragma unroll
      for (int k = 0; k < 32; ++k)
        w[k] = pack_bf16x2(pr[2 * k] * (__uint_as_float(x[2 * k]) - Drow),
                           pr[2 * k + 1] * (__uint_as_float(x[2 * k + 1]) - Drow));
      // dS packed into the first 32 of this warpgroup's own 64 dP columns
      tmem_st32(buf, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
      if (lane == 0) LAGA_TRACE_POINT(dq, 11, j);
    }
    if (ok && warp_wait(dq_done, 0, 82)) {
      LAGA_TRACE_POINT(dq, 29, 0);
      tc_fence_after();
      // Epilogue: dq (scaled, bf16) through shared memory and tensor-map stores,
      // which the TMA unit carries out while the CTA ends. Every MMA has finished,
      // so the Q tile's space is free: each warp stages its 32 rows x 96 columns
      // as three [32 rows][64 B] boxes (64-byte swizzle); rows past Sq are clipped
      // by the map.
      uint8_t* stage = smem + OFF_Q + (warp - 2) * 6144;
#pragma unroll 1
      for (int j = 0; j < 3; ++j) {
        const int c = 3 * half + j;
        uint32_t u[32];
        tmem_ld32(tmem + COL_DQ + lane_off + c * 32, u);  // warp-collective: every lane takes part
        tmem_wait_ld();
        uint8_t* box = stage + j * 2048;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 o;
          o.x = pack_bf16x2(__uint_as_float(u[8 * v + 0]) * p.scale, __uint_as_float(u[8 * v + 1]) * p.scale);
          o.y = pack_bf16x2(__uint_as_float(u[8 * v + 2]) * p.scale, __uint_as_float(u[8 * v + 3]) * p.scale);
          o.z = pack_bf16x2(__uint_as_float(u[8 * v + 4]) * p.scale, __uint_as_float(u[8 * v + 5]) * p.scale);
          o.w = pack_bf16x2(__uint_as_float(u[8 * v + 6]) * p.scale, __uint_as_float(u[8 * v + 7]) * p.scale);
          *reinterpret_cast<uint4*>(box + sw64_offset(lane, v)) = o;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < 3; ++j) tma_store_3d(&mdQ, stage + j * 2048, h * 192 + 32 * (3 * half + j), t * BQ + quarter * 32, b);
        bulk_commit_group();
        bulk_wait_read_all();  // shared memory must not go away under a store
      }
      __syncwarp();
    }
  }

  LAGA_TRACE_POINT(dq, 28, 0);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) publish_abort(abort_flag, p.status);
  LAGA_TRACE_POINT(dq, 31, 0);
  LAGA_TRACE_CTA_END(dq);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

LaunchResult tc_attn_bwd_dq(const Dims& d, const bf16* q, const bf16* k_rope, const bf16* dout,
                            const BwdWorkspace& w, bf16* dq, cudaStream_t st) {
  LaunchResult r;
  CUtensorMap mQ, mK, mR, mV;
  const uint32_t qbox[3] = {64, BQ, 1};
  {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 192;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    r.cu = make_tmap(&mQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t kv_inner = static_cast<uint64_t>(d.n_h) * 128;
  const uint64_t kv_rows = static_cast<uint64_t>(d.B) * d.skv_pad;
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[2] = {kv_inner, kv_rows};
    const uint64_t strides[1] = {kv_inner * 2};
    const uint32_t box[2] = {64, BKV};
    r.cu = make_tmap(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.k_ws, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    if (r.cu == CUDA_SUCCESS)
      r.cu = make_tmap(&mV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.v_ws, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(d.S), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(d.S) * 128};
    const uint32_t box[3] = {64, BKV, 1};
    r.cu = make_tmap(&mR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_rope, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  CUtensorMap mdQ;  // dq's [32 rows][32] boxes, 3D over [B][Sq][n_h*192]: rows past Sq clip
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 192;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    const uint32_t box[3] = {32, 32, 1};
    r.cu = make_tmap(&mdQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
  }
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps attention backward (dq)";
    return r;
  }
  Params p{};
  p.status = device_status_ptr();
  p.Sq = d.Sq;
  p.S = d.S;
  p.n_h = d.n_h;
  p.q_offset = d.q_offset;
  p.q_split = d.q_split;
  p.q_offset2 = d.q_offset2;
  p.causal = d.causal ? 1 : 0;
  p.skv_pad = d.skv_pad;
  p.sq_pad = d.sq_pad;
  p.n_q_tiles = (d.Sq + BQ - 1) / BQ;
  p.scale = d.scale;
  p.scale_log2 = d.scale * 1.4426950408889634f;
  p.lse2 = w.lse2;
  p.delta = w.delta;
  p.dout = dout;
  r.err = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(attn_bwd_dq)";
    return r;
  }
  attn_bwd_dq_kernel<<<dim3(p.n_q_tiles, d.n_h, d.B), NTHREADS, SMEM_BYTES, st>>>(mQ, mK, mR, mV, mdQ, p);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "attn_bwd_dq_kernel launch";
  return r;
}

}  // namespace laga
