// Attention backward, query side: dq on the tensor cores (d_qk = 128 + 64,
// d_v = 128, bf16 operands, fp32 accumulation).
//
// One CTA per (128-row query tile, head, batch element); it walks the 64-row
// key tiles the tile can see and keeps the whole dq tile (192 head dims) in
// TMEM, so every dq element is written once, with no accumulation in memory:
//   S  = Q K^T          P  = exp(S * scale - lse)      (lse from the forward)
//   dP = dO V^T         dS = P o (dP - D)
//   dq += dS K          (scale applied once at the end)
// dS is written back into TMEM as packed bf16 over S and feeds the dq product
// as the A operand straight from TMEM. The RoPE-key concat is folded in as in
// the forward: S = Q_nope K_nope^T + Q_rope k_rope^T, and dq's last 64 columns
// come from the k_rope tile.
//
// Warp roles (352 threads):
//   warp 0      lane 0: TMA for Q and dO once, then key tiles
//   warp 1      TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 2..9  two warpgroups; each thread owns one query row (TMEM lane) and
//               half of the tile's 64 key columns: P, dS, and half the epilogue
//   warp 10     lane 0: TMA for value tiles (its own warp, so that its waits
//               never hold back the key-tile producer)
// TMEM columns: S/dS x2 [0,128), dP x2 [128,256), dq [256,448), dO [448,512).
// dO is the same for every key tile: the query-row warps copy it into TMEM
// once and dP = dO V^T reads it from there (A operand from TMEM), which takes
// its reads off the shared-memory port that bounds this kernel.
#include "internal.h"
#include "ptx.cuh"

LAGA_TRACE_DEFINE(dq)

namespace laga {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 64;
constexpr int NSTAGE = 3;
constexpr int QBOX = 16384;  // [128 rows][64] bf16
constexpr int KBOX = 8192;   // [64 rows][64] bf16
constexpr int Q_BYTES = 3 * QBOX;
constexpr int DO_BYTES = 2 * QBOX;
constexpr int K_BYTES = 3 * KBOX;
constexpr int V_BYTES = 2 * KBOX;
constexpr int OFF_Q = 0;
constexpr int OFF_DO = OFF_Q + Q_BYTES;
constexpr int OFF_K = OFF_DO + DO_BYTES;
constexpr int OFF_V = OFF_K + NSTAGE * K_BYTES;
constexpr int OFF_BARS = OFF_V + NSTAGE * V_BYTES;
constexpr int SMEM_BYTES = OFF_BARS + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 256, COL_DO = 448;
constexpr uint32_t IDESC_S = idesc_bf16(128, 64, false, false);
constexpr uint32_t IDESC_DQ = idesc_bf16(128, 192, false, true);
constexpr int NTHREADS = 352;
constexpr uint32_t SOFTMAX_WARPS = 8;

struct Params {
  int* status;
  int Sq, S, n_h, q_offset, causal, skv_pad, sq_pad, n_q_tiles;
  float scale, scale_log2;
  const float* lse2;
  const float* delta;
  bf16* dq;
};

// TMEM column of packed bf16 chunk k (16 keys) of a 64-key tile: the two
// warpgroups pack their halves at columns [0,16) and [32,48).
__device__ __forceinline__ uint32_t packed_col(int k) { return 8u * k + 16u * (k >> 1); }

__device__ __forceinline__ int n_kv_tiles(const Params& p, int t) {
  const int last = p.causal ? p.q_offset + min(p.Sq, (t + 1) * BQ) - 1 : p.S - 1;
  return last / BKV + 1;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                       const __grid_constant__ CUtensorMap mR, const __grid_constant__ CUtensorMap mV,
                       const __grid_constant__ CUtensorMap mdO, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  LAGA_TRACE_CTA_BEGIN(dq);
  LAGA_TRACE_POINT(dq, 30, 0);
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [NSTAGE]
  uint64_t* k_empty = bars + 4;  // [NSTAGE]
  uint64_t* v_full = bars + 7;   // [NSTAGE]
  uint64_t* v_empty = bars + 10; // [NSTAGE]
  uint64_t* s_full = bars + 13;  // [2]  S(j) and dP(j) done
  uint64_t* ds_full = bars + 15; // [2]  dS(j) in TMEM
  uint64_t* dq_done = bars + 17;
  uint64_t* drain = bars + 18;
  uint64_t* do_tmem = bars + 19;  // dO copied into TMEM by the query-row warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = p.n_q_tiles - 1 - static_cast<int>(blockIdx.x);  // heaviest tiles first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int n_kv = n_kv_tiles(p, t);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&ds_full[i], SOFTMAX_WARPS);
    }
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
      tma_prefetch_desc(&mdO);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mR);
      mbar_arrive_expect_tx(q_full, Q_BYTES + DO_BYTES);
      const int q0 = t * BQ;
      tma_load_3d(smem + OFF_Q, &mQ, q_full, h * 192, q0, b);
      tma_load_3d(smem + OFF_Q + QBOX, &mQ, q_full, h * 192 + 64, q0, b);
      tma_load_3d(smem + OFF_Q + 2 * QBOX, &mQ, q_full, h * 192 + 128, q0, b);
      tma_load_3d(smem + OFF_DO, &mdO, q_full, h * 128, q0, b);
      tma_load_3d(smem + OFF_DO + QBOX, &mdO, q_full, h * 128 + 64, q0, b);
      int j = 0;
      for (; j < n_kv; ++j) {
        const int s = j % NSTAGE;
        if (!mbar_wait_or_abort(&k_empty[s], ((j / NSTAGE) & 1) ^ 1, abort_flag, 71)) break;
        uint8_t* dst = smem + OFF_K + s * K_BYTES;
        mbar_arrive_expect_tx(&k_full[s], K_BYTES);
        const int row = b * p.skv_pad + j * BKV;
        tma_load_2d(dst, &mK, &k_full[s], h * 128, row);
        tma_load_2d(dst + KBOX, &mK, &k_full[s], h * 128 + 64, row);
        tma_load_3d(dst + 2 * KBOX, &mR, &k_full[s], 0, j * BKV, b);
      }
      if (j < n_kv) {
        mbar_drain(q_full, 0);
        for (int i = j - NSTAGE < 0 ? 0 : j - NSTAGE; i < j; ++i)
          mbar_drain(&k_full[i % NSTAGE], (i / NSTAGE) & 1);
      }
    }
  } else if (warp == 10) {
    if (lane == 0) {
      tma_prefetch_desc(&mV);
      int j = 0;
      for (; j < n_kv; ++j) {
        const int s = j % NSTAGE;
        if (!mbar_wait_or_abort(&v_empty[s], ((j / NSTAGE) & 1) ^ 1, abort_flag, 72)) break;
        uint8_t* dst = smem + OFF_V + s * V_BYTES;
        mbar_arrive_expect_tx(&v_full[s], V_BYTES);
        const int row = b * p.skv_pad + j * BKV;
        tma_load_2d(dst, &mV, &v_full[s], h * 128, row);
        tma_load_2d(dst + KBOX, &mV, &v_full[s], h * 128 + 64, row);
      }
      if (j < n_kv)
        for (int i = j - NSTAGE < 0 ? 0 : j - NSTAGE; i < j; ++i)
          mbar_drain(&v_full[i % NSTAGE], (i / NSTAGE) & 1);
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop; an elected lane issues. Each barrier is
    // tested (without blocking) before the MMA group that precedes its use, so the
    // check after that group costs no shared-memory round trip behind the MMAs.
    bool ok = warp_wait_or_abort(q_full, 0, abort_flag, 73) && warp_wait_or_abort(do_tmem, 0, abort_flag, 77);
    bool issued = false;
    tc_fence_after();
    const uint64_t q_desc = sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
    auto issue_s = [&](int j) {  // S(j) = Q K_j^T
      const uint64_t k_desc = sdesc_sw128(smem_u32(smem + OFF_K + (j % NSTAGE) * K_BYTES), 16, 1024);
      const uint32_t ds = tmem + COL_S + 64u * (j & 1);
#pragma unroll
      for (int kk = 0; kk < 12; ++kk) {
        const uint32_t c = kk >> 2, k = kk & 3;
        mma_ss_warp(ds, q_desc + ((c * QBOX + k * 32) >> 4), k_desc + ((c * KBOX + k * 32) >> 4), IDESC_S,
                    kk > 0 ? 1u : 0u);
      }
    };
    auto issue_dp = [&](int j) {  // dP(j) = dO V_j^T, then S(j) and dP(j) are announced
      const int s = j % NSTAGE;
      const uint64_t v_desc = sdesc_sw128(smem_u32(smem + OFF_V + s * V_BYTES), 16, 1024);
      const uint32_t dd = tmem + COL_DP + 64u * (j & 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // head dims [16kk, 16kk + 16): dO columns [8kk, 8kk + 8)
        mma_ts_warp(dd, tmem + COL_DO + kk * 8, v_desc + (((kk >> 2) * KBOX + (kk & 3) * 32) >> 4), IDESC_S,
                    kk > 0 ? 1u : 0u);
      mma_commit_warp(&s_full[j & 1]);
      mma_commit_warp(&v_empty[s]);
    };
    auto issue_dq = [&](int j) {  // dq += dS(j) K_j : A = dS (TMEM, packed bf16), B = key tile MN-major (N = 192)
      const int s = j % NSTAGE;
      const uint64_t k_mn = sdesc_sw128(smem_u32(smem + OFF_K + s * K_BYTES), KBOX, 1024);
      const uint32_t ds = tmem + COL_S + 64u * (j & 1);
#pragma unroll
      for (int k = 0; k < BKV / 16; ++k)
        mma_ts_warp(tmem + COL_DQ, ds + packed_col(k), k_mn + ((k * 2048) >> 4), IDESC_DQ, (j > 0 || k > 0) ? 1u : 0u);
      mma_commit_warp(&k_empty[s]);
    };
    // One loop issues everything, the first step included, so that every MMA group
    // exists once in the binary: code run once per CTA falls out of the
    // instruction cache between CTAs and then issues several times slower.
    // Iteration j: S(j+1), dP(j+1) (j+1 < n), then dq(j) (j >= 0); S and dP of
    // j+1 go ahead of dq(j) so that the softmax of j+1 overlaps dq(j).
    uint32_t tk = 0;
    for (int j = -1; j < n_kv && ok; ++j) {
      const uint32_t dph = (j >> 1) & 1;
      uint32_t td = 0;
      if (j + 1 < n_kv) {
        const int jn = j + 1, sn = jn % NSTAGE;
        const uint32_t pn = (jn / NSTAGE) & 1;
        if (!warp_wait_token(&k_full[sn], pn, tk, abort_flag, 74)) { ok = false; break; }
        const uint32_t tv = mbar_test(&v_full[sn], pn);
        tc_fence_after();
        issue_s(jn);
        issued = true;
        if (!warp_wait_token(&v_full[sn], pn, tv, abort_flag, 75)) { ok = false; break; }
        if (j >= 0) td = mbar_test(&ds_full[j & 1], dph);
        tc_fence_after();
        issue_dp(jn);
      } else if (j >= 0) {
        td = mbar_test(&ds_full[j & 1], dph);
      }
      if (j >= 0) {
        if (!warp_wait_token(&ds_full[j & 1], dph, td, abort_flag, 76)) { ok = false; break; }
        tk = j + 2 < n_kv ? mbar_test(&k_full[(j + 2) % NSTAGE], ((j + 2) / NSTAGE) & 1) : 1u;
        tc_fence_after();
        issue_dq(j);
      } else {
        tk = n_kv > 1 ? mbar_test(&k_full[1 % NSTAGE], (1 / NSTAGE) & 1) : 1u;
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
    const int half = (warp - 2) >> 2;  // warpgroup: key columns [32*half, 32*half + 32)
    const int r = quarter * 32 + lane;
    const int q_row = t * BQ + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int limit = p.causal ? p.q_offset + q_row : p.S - 1;  // last visible key
    const long long roff = (static_cast<long long>(b) * p.n_h + h) * p.sq_pad + q_row;
    const float lse2 = p.lse2[roff];  // +inf on padded rows: P = 0 there
    const float Drow = p.delta[roff];
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
      const bool all = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      __syncwarp();  // order lane 0's acquire before the other lanes' reads
      return all;
    };
    // dO row r -> TMEM lane r as packed bf16 pairs; warpgroup `half` copies
    // head dims [64*half, 64*half + 64) (box `half` of the swizzled TMA tile).
    if (!warp_wait(q_full, 0, 83)) ok = false;
    if (ok) {
      uint32_t w[32];
      const uint8_t* box = smem + OFF_DO + half * QBOX;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = *reinterpret_cast<const uint4*>(box + sw128_offset(r, k));
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
      if (!warp_wait(&s_full[j & 1], (j >> 1) & 1, 81)) { ok = false; break; }
      if (lane == 0) LAGA_TRACE_POINT(dq, 10, j);
      tc_fence_after();
      const uint32_t s_addr = tmem + COL_S + 64u * (j & 1) + lane_off;
      const uint32_t dp_addr = tmem + COL_DP + 64u * (j & 1) + lane_off;
      const int kv_first = j * BKV + 32 * half;  // this thread's first key column
      uint32_t us[32], ud[32], w[16];
      tmem_ld32(s_addr + 32 * half, us);
      tmem_ld32(dp_addr + 32 * half, ud);
      tmem_wait_ld();
      if (kv_first + 31 <= limit) {  // every key of the half-tile visible
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(us[2 * k]), p.scale_log2, -lse2));
          const float p1 = ex2_approx(fmaf(__uint_as_float(us[2 * k + 1]), p.scale_log2, -lse2));
          w[k] = pack_bf16x2(p0 * (__uint_as_float(ud[2 * k]) - Drow), p1 * (__uint_as_float(ud[2 * k + 1]) - Drow));
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const bool v0 = kv_first + 2 * k <= limit, v1 = kv_first + 2 * k + 1 <= limit;
          const float p0 = v0 ? ex2_approx(fmaf(__uint_as_float(us[2 * k]), p.scale_log2, -lse2)) : 0.f;
          const float p1 = v1 ? ex2_approx(fmaf(__uint_as_float(us[2 * k + 1]), p.scale_log2, -lse2)) : 0.f;
          w[k] = pack_bf16x2(p0 * (__uint_as_float(ud[2 * k]) - Drow), p1 * (__uint_as_float(ud[2 * k + 1]) - Drow));
        }
      }
      // dS packed in place over this half's own score columns (key pair k -> column 32*half + k),
      // so the other warpgroup's scores are never overwritten before it has read them
      tmem_st16(s_addr + 32 * half, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[j & 1]);
      if (lane == 0) LAGA_TRACE_POINT(dq, 11, j);
    }
    if (ok && warp_wait(dq_done, 0, 82)) {
      LAGA_TRACE_POINT(dq, 29, 0);
      tc_fence_after();
      const bool valid = q_row < p.Sq;
      bf16* dst = p.dq + ((static_cast<long long>(b) * p.Sq + q_row) * p.n_h + h) * 192;
#pragma unroll 1
      for (int c = 3 * half; c < 3 * half + 3; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + COL_DQ + lane_off + c * 32, u);  // warp-collective: every lane takes part
        tmem_wait_ld();
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(u[8 * v + 0]) * p.scale, __uint_as_float(u[8 * v + 1]) * p.scale);
            o.y = pack_bf16x2(__uint_as_float(u[8 * v + 2]) * p.scale, __uint_as_float(u[8 * v + 3]) * p.scale);
            o.z = pack_bf16x2(__uint_as_float(u[8 * v + 4]) * p.scale, __uint_as_float(u[8 * v + 5]) * p.scale);
            o.w = pack_bf16x2(__uint_as_float(u[8 * v + 6]) * p.scale, __uint_as_float(u[8 * v + 7]) * p.scale);
            d4[v] = o;
          }
        }
      }
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
  CUtensorMap mQ, mK, mR, mV, mdO;
  const uint32_t qbox[3] = {64, BQ, 1};
  {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 192;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    r.cu = make_tmap(&mQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 128;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    r.cu = make_tmap(&mdO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dout, dims, strides, qbox,
                     CU_TENSOR_MAP_SWIZZLE_128B);
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
  p.causal = d.causal ? 1 : 0;
  p.skv_pad = d.skv_pad;
  p.sq_pad = d.sq_pad;
  p.n_q_tiles = (d.Sq + BQ - 1) / BQ;
  p.scale = d.scale;
  p.scale_log2 = d.scale * 1.4426950408889634f;
  p.lse2 = w.lse2;
  p.delta = w.delta;
  p.dq = dq;
  r.err = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(attn_bwd_dq)";
    return r;
  }
  attn_bwd_dq_kernel<<<dim3(p.n_q_tiles, d.n_h, d.B), NTHREADS, SMEM_BYTES, st>>>(mQ, mK, mR, mV, mdO, p);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "attn_bwd_dq_kernel launch";
  return r;
}

}  // namespace laga
