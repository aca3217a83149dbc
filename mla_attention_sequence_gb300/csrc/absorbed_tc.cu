// Attention in latent space for the absorbed MLA form (the variant LAGA
// rejects), on the tensor cores. Run for comparison only; the library's own
// forward is the explicit form with K/V rebuilt per head.
//
// "A Training-Memory Regression in MLA Sequence Parallelism ... LAGA"
// (weekinpapers page, Abstract): the absorbed form folds W_UK into the query and
// attends in the latent space, which is what inference decode uses. For head h:
//   q_abs  = [q_nope_h W_UK_h^T | q_rope_h]            (d_c + d_rope = 576 wide)
//   s_ij   = scale * q_abs_i . [c_kv_j | k_rope_j]     (one key for every head)
//   ctx_i  = sum_j softmax_j(s_ij) c_kv_j              (d_c = 512 wide)
//   out_i  = ctx_i W_UV_h
// The scores equal the explicit form's (q_nope W_UK^T c_kv^T = q_nope K_nope^T),
// so scale and lse are the explicit form's. This kernel is the middle line;
// the two projections are tensor-core GEMMs (gemm_tc.cu, QLAT and OUTPROJ).
//
// One CTA per (128-row query tile, head, batch element, value half): TMEM
// cannot hold a 128 x 512 fp32 context tile next to the scores, so each CTA
// accumulates 256 of the 512 context columns and computes the scores itself.
// Keys stream in 64-row tiles of [c_kv | k_rope] (nine [64 x 64] boxes, 72 KB);
// the query tile (nine [128 x 64] boxes, 144 KB) stays in shared memory.
// The per-tile order is serial: load tile j, S(j) = Q K_j^T (36 K16 steps,
// N = 64), online softmax, O += P(j) V_j (the value half of the same boxes read
// MN-major, N = 256); the next tile loads once PV(j) has read the buffer.
//
// Warp roles (192 threads): warp 0 lane 0 TMA; warp 1 TMEM allocation and the
// MMA issue loop; warps 2..5 softmax, one query row per thread (TMEM lane).
// TMEM columns: S/P [0,64) (and [64,128) for odd tiles), O [256,512).
#include "internal.h"
#include "ptx.cuh"

namespace laga {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 64;
constexpr int NBOX = 9;        // 8 latent boxes + 1 RoPE box
constexpr int QBOX = 16384;    // [128 rows][64] bf16
constexpr int KBOX = 8192;     // [64 rows][64] bf16
constexpr int Q_BYTES = NBOX * QBOX;
constexpr int K_BYTES = NBOX * KBOX;
constexpr int SMEM_BYTES = Q_BYTES + K_BYTES + 1024 + 256;
constexpr int NTHREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 256;
constexpr int DV_HALF = 256;
constexpr uint32_t IDESC_S = idesc_bf16(128, BKV, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, DV_HALF, false, true);
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Params {
  int* status;
  int Sq, S, n_h, q_offset, causal, n_q_tiles;
  float scale_log2;
  bf16* ctx;   // [B*Sq][n_h*512]
  float* lse;  // [B][n_h][Sq]
};

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_absorbed_kernel(const __grid_constant__ CUtensorMap mQl, const __grid_constant__ CUtensorMap mQr,
                         const __grid_constant__ CUtensorMap mC, const __grid_constant__ CUtensorMap mR,
                         const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + Q_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Q_BYTES + K_BYTES);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 2;  // PV(j) done: the key tile buffer may be refilled
  uint64_t* s_full = bars + 3;
  uint64_t* p_full = bars + 4;
  uint64_t* drain = bars + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = p.n_q_tiles - 1 - static_cast<int>(blockIdx.x);  // heaviest tiles first
  const int vh = blockIdx.y & 1;                                 // value half
  const int h = blockIdx.y >> 1;
  const int b = blockIdx.z;
  const int last_key = p.causal ? p.q_offset + min(p.Sq, (t + 1) * BQ) - 1 : p.S - 1;
  const int n_kv = last_key / BKV + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
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
      tma_prefetch_desc(&mQl);
      tma_prefetch_desc(&mC);
      mbar_arrive_expect_tx(q_full, Q_BYTES);
      for (int c = 0; c < 8; ++c) tma_load_3d(sQ + c * QBOX, &mQl, q_full, h * 512 + c * 64, t * BQ, b);
      tma_load_3d(sQ + 8 * QBOX, &mQr, q_full, h * 192 + 128, t * BQ, b);
      int j = 0;
      for (; j < n_kv; ++j) {
        if (j > 0 && !mbar_wait_or_abort(kv_empty, (j - 1) & 1, abort_flag, 201)) break;
        mbar_arrive_expect_tx(kv_full, K_BYTES);
        for (int c = 0; c < 8; ++c) tma_load_3d(sK + c * KBOX, &mC, kv_full, c * 64, j * BKV, b);
        tma_load_3d(sK + 8 * KBOX, &mR, kv_full, 0, j * BKV, b);
      }
      if (j < n_kv) {  // aborted: let the copies in flight land
        mbar_drain(q_full, 0);
        if (j > 0) mbar_drain(kv_full, (j - 1) & 1);
      }
    }
  } else if (warp == 1) {
    bool ok = warp_wait_or_abort(q_full, 0, abort_flag, 202);
    bool issued = false;
    const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
    // the value half of the key tile, MN-major: 64-column atoms 8 KB apart
    const uint64_t v_desc = sdesc_sw128(smem_u32(sK + vh * 4 * KBOX), KBOX, 1024);
    for (int j = 0; j < n_kv && ok; ++j) {
      if (!warp_wait_or_abort(kv_full, j & 1, abort_flag, 203)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sbuf = tmem + static_cast<uint32_t>(j & 1) * BKV;
#pragma unroll
      for (int c = 0; c < NBOX; ++c) {  // dims [64c, 64c + 64): four K16 steps in box c
        const uint64_t a = q_desc + ((c * QBOX) >> 4), k = k_desc + ((c * KBOX) >> 4);
        mma4_ss_warp(sbuf, a, a + 2, a + 4, a + 6, k, k + 2, k + 4, k + 6, IDESC_S, c > 0 ? 1u : 0u);
      }
      issued = true;
      mma_commit_warp(s_full);
      if (!warp_wait_or_abort(p_full, j & 1, abort_flag, 204)) { ok = false; break; }
      tc_fence_after();
      // O += P V : A = P (TMEM, packed bf16, 32 columns), B = value half (keys x 256)
      mma4_ts_warp(tmem + COL_O, sbuf, sbuf + 8, sbuf + 16, sbuf + 24, v_desc, v_desc + (2048 >> 4),
                   v_desc + (4096 >> 4), v_desc + (6144 >> 4), IDESC_PV, j > 0 ? 1u : 0u);
      mma_commit_warp(kv_empty);
    }
    if (!ok && issued) {
      mma_commit_warp(drain);
      if (lane == 0) mbar_drain(drain, 0);
      __syncwarp();
    }
  } else {
    // ---------------- softmax: thread owns query row r of the tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int q_row = t * BQ + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int limit = p.causal ? p.q_offset + q_row : p.S - 1;  // last visible key
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
      const bool all = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      __syncwarp();
      return all;
    };
    for (int j = 0; j < n_kv && ok; ++j) {
      if (!warp_wait(s_full, j & 1, 205)) { ok = false; break; }
      tc_fence_after();
      const uint32_t s_addr = tmem + static_cast<uint32_t>(j & 1) * BKV + lane_off;
      uint32_t x[64];
      tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(x));
      tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
      tmem_wait_ld();
      const int kv0 = j * BKV;
      if (kv0 + BKV - 1 > limit) {
#pragma unroll
        for (int i = 0; i < BKV; ++i)
          if (kv0 + i > limit) x[i] = 0xff800000u;  // -inf
      }
      float mx = __uint_as_float(x[0]);
#pragma unroll
      for (int i = 1; i < BKV; ++i) mx = fmaxf(mx, __uint_as_float(x[i]));
      const float mt = mx * sl2;
      float m_use = m_run, alpha = 1.f;
      bool rescale = false;
      if (m_run == -INFINITY) {
        m_use = mt;
      } else if (mt > m_run + RESCALE_THRESHOLD) {
        m_use = mt;
        alpha = ex2_approx(m_run - mt);
        rescale = true;
      }
      const float neg_m = m_use == -INFINITY ? 0.f : -m_use;
      float sum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(x[2 * i]), sl2, neg_m));
        const float p1 = ex2_approx(fmaf(__uint_as_float(x[2 * i + 1]), sl2, neg_m));
        sum += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + sum;
      m_run = m_use;
      tmem_st32(s_addr, pk);
      if (__any_sync(0xffffffffu, rescale)) {
        // PV(j-1) is complete: tile j was loaded only after it had read its buffer
        const uint32_t o_addr = tmem + COL_O + lane_off;
#pragma unroll 1
        for (int c = 0; c < DV_HALF / 32; ++c) {
          uint32_t u[32];
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
      if (lane == 0) mbar_arrive(p_full);
    }
    // the last PV is done once the producer's last empty phase completes
    if (ok && warp_wait(kv_empty, (n_kv - 1) & 1, 206)) {
      tc_fence_after();
      const bool valid = q_row < p.Sq;
      const float inv = 1.f / l_run;
      const uint32_t o_addr = tmem + COL_O + lane_off;
      bf16* orow = p.ctx + (static_cast<long long>(b) * p.Sq + q_row) * (static_cast<long long>(p.n_h) * 512) +
                   h * 512 + vh * DV_HALF;
#pragma unroll 1
      for (int c = 0; c < DV_HALF / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(o_addr + c * 32, u);
        tmem_wait_ld();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(u[8 * v + 0]) * inv, __uint_as_float(u[8 * v + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(u[8 * v + 2]) * inv, __uint_as_float(u[8 * v + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(u[8 * v + 4]) * inv, __uint_as_float(u[8 * v + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(u[8 * v + 6]) * inv, __uint_as_float(u[8 * v + 7]) * inv);
            dst[v] = w;
          }
        }
      }
      if (valid && vh == 0)
        p.lse[(static_cast<long long>(b) * p.n_h + h) * p.Sq + q_row] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) publish_abort(abort_flag, p.status);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

LaunchResult tc_absorbed_attn(const Dims& d, const bf16* q_lat, const bf16* q, const bf16* c_kv, const bf16* k_rope,
                              bf16* ctx, float* lse, cudaStream_t st) {
  LaunchResult r;
  CUtensorMap mQl, mQr, mC, mR;
  {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 512;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    const uint32_t box[3] = {64, BQ, 1};
    r.cu = make_tmap(&mQl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q_lat, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 192;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    const uint32_t box[3] = {64, BQ, 1};
    r.cu = make_tmap(&mQr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[3] = {512, static_cast<uint64_t>(d.S), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {1024, static_cast<uint64_t>(d.S) * 1024};
    const uint32_t box[3] = {64, BKV, 1};
    r.cu = make_tmap(&mC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c_kv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(d.S), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(d.S) * 128};
    const uint32_t box[3] = {64, BKV, 1};
    r.cu = make_tmap(&mR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_rope, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps absorbed attention";
    return r;
  }
  Params p{};
  p.status = device_status_ptr();
  p.Sq = d.Sq;
  p.S = d.S;
  p.n_h = d.n_h;
  p.q_offset = d.q_offset;
  p.causal = d.causal ? 1 : 0;
  p.n_q_tiles = (d.Sq + BQ - 1) / BQ;
  p.scale_log2 = d.scale * 1.4426950408889634f;
  p.ctx = ctx;
  p.lse = lse;
  r.err = cudaFuncSetAttribute(attn_absorbed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(attn_absorbed)";
    return r;
  }
  attn_absorbed_kernel<<<dim3(p.n_q_tiles, 2 * d.n_h, d.B), NTHREADS, SMEM_BYTES, st>>>(mQl, mQr, mC, mR, p);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "attn_absorbed_kernel launch";
  return r;
}

}  // namespace laga
