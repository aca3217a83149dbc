// Forward attention with the K/V reconstruction fused in: each CTA rebuilds
// the no-RoPE key and value tiles of its head from the latent tile on the
// tensor cores, instead of reading K_nope / V that a separate GEMM
// materialised in HBM (LAGA: per-head K/V rebuilt locally from the gathered
// latent, here tile by tile inside the attention kernel).
//
// One CTA per (128-row query tile, head, batch element). Per 128-row key tile j:
//   Kacc = c_kv_j W_UK_h, Vacc = c_kv_j W_UV_h   (K = d_c = 512, into TMEM)
//   convert: Kacc, Vacc -> bf16 shared-memory operand tiles (128-byte swizzle)
//   S = Q [K_nope | k_rope]^T, online softmax, O += P V      (as the plain forward)
// The rebuild costs 2 * 128 * 512 * 256 flops per key tile against
// 2 * 128 * 128 * 320 for the attention itself, so the tensor cores do about
// 4.2x the plain forward's work; what it saves is the K/V round trip through HBM.
//
// Warp roles (320 threads):
//   warp 0      lane 0: TMA ring of latent / weight chunks; lane 1: Q and k_rope tiles
//   warp 1      TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 2..5  softmax (one query row per thread) and the epilogue
//   warps 6..9  convert (one key row per thread)
// TMEM columns: S/P [0,128), O [128,256), Kacc [256,384), Vacc [384,512).
// MMA order S(j), rebuild(j+1), PV(j): the rebuild of the next tile runs while
// softmax works on this one.
#include "internal.h"
#include "ptx.cuh"

namespace laga {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int BOX = 16384;   // [128 rows][64] bf16
constexpr int WBOX = 8192;   // [64 rows][64] bf16
constexpr int NCHUNK = 8;    // d_c / 64
constexpr int STAGES = 2;
constexpr int Q_BYTES = 3 * BOX;
constexpr int CHUNK_BYTES = BOX + 4 * WBOX;  // latent chunk + W_UK chunk + W_UV chunk
constexpr int K_BYTES = 3 * BOX;
constexpr int V_BYTES = 2 * BOX;
constexpr int OFF_Q = 0;
constexpr int OFF_RING = OFF_Q + Q_BYTES;
constexpr int OFF_K = OFF_RING + STAGES * CHUNK_BYTES;
constexpr int OFF_V = OFF_K + K_BYTES;
constexpr int OFF_BARS = OFF_V + V_BYTES;
constexpr int SMEM_BYTES = OFF_BARS + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 128, COL_KA = 256, COL_VA = 384;
constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 128, false, true);
constexpr uint32_t IDESC_RC = idesc_bf16(128, 128, false, true);
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr int NTHREADS = 320;

struct Params {
  int* status;
  int Sq, S, n_h, q_offset, causal, n_q_tiles;
  float scale_log2;
  bf16* out;
  float* lse;
};

__device__ __forceinline__ int n_kv_tiles(const Params& p, int t) {
  const int last = p.causal ? p.q_offset + min(p.Sq, (t + 1) * BQ) - 1 : p.S - 1;
  return last / BKV + 1;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd_fused_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mC,
                          const __grid_constant__ CUtensorMap mWK, const __grid_constant__ CUtensorMap mWV,
                          const __grid_constant__ CUtensorMap mR, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* q_full = bars + 0;
  uint64_t* st_full = bars + 1;    // [STAGES]
  uint64_t* st_empty = bars + 3;   // [STAGES]
  uint64_t* acc_full = bars + 5;   // rebuild of a tile done (Kacc, Vacc)
  uint64_t* acc_free = bars + 6;   // Kacc, Vacc read out by the convert warps
  uint64_t* kt_full = bars + 7;    // K_nope / V operand tiles written
  uint64_t* rope_full = bars + 8;  // k_rope tile landed
  uint64_t* kv_free = bars + 9;    // S and PV of a tile done: operand tiles reusable
  uint64_t* s_full = bars + 10;
  uint64_t* p_full = bars + 11;
  uint64_t* o_done = bars + 12;
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = p.n_q_tiles - 1 - static_cast<int>(blockIdx.x);
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int n_kv = n_kv_tiles(p, t);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&st_full[i], 1);
      mbar_init(&st_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_free, 4);
    mbar_init(kt_full, 4);
    mbar_init(rope_full, 1);
    mbar_init(kv_free, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
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

  auto warp_wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    bool w = true;
    if (lane == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
    const bool all = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    __syncwarp();  // order lane 0's acquire before the other lanes' reads
    return all;
  };

  if (warp == 0) {
    if (lane == 0) {
      // latent / weight chunk ring: tile j, chunk c covers latent columns [64c, 64c + 64)
      tma_prefetch_desc(&mC);
      tma_prefetch_desc(&mWK);
      tma_prefetch_desc(&mWV);
      int it = 0;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        for (int c = 0; c < NCHUNK; ++c, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_or_abort(&st_empty[s], ((it / STAGES) & 1) ^ 1, abort_flag, 91)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + OFF_RING + s * CHUNK_BYTES;
          mbar_arrive_expect_tx(&st_full[s], CHUNK_BYTES);
          tma_load_3d(dst, &mC, &st_full[s], c * 64, j * BKV, b);
          tma_load_2d(dst + BOX, &mWK, &st_full[s], h * 128, c * 64);
          tma_load_2d(dst + BOX + WBOX, &mWK, &st_full[s], h * 128 + 64, c * 64);
          tma_load_2d(dst + BOX + 2 * WBOX, &mWV, &st_full[s], h * 128, c * 64);
          tma_load_2d(dst + BOX + 3 * WBOX, &mWV, &st_full[s], h * 128 + 64, c * 64);
        }
      }
      if (!ok) {
        const int first = it > STAGES ? it - STAGES : 0;
        for (int k = first; k < it; ++k) mbar_drain(&st_full[k % STAGES], (k / STAGES) & 1);
      }
    } else if (lane == 1) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mR);
      mbar_arrive_expect_tx(q_full, Q_BYTES);
      tma_load_3d(smem + OFF_Q, &mQ, q_full, h * 192, t * BQ, b);
      tma_load_3d(smem + OFF_Q + BOX, &mQ, q_full, h * 192 + 64, t * BQ, b);
      tma_load_3d(smem + OFF_Q + 2 * BOX, &mQ, q_full, h * 192 + 128, t * BQ, b);
      int j = 0;
      for (; j < n_kv; ++j) {
        if (j > 0 && !mbar_wait_or_abort(kv_free, (j - 1) & 1, abort_flag, 92)) break;
        mbar_arrive_expect_tx(rope_full, BOX);
        tma_load_3d(smem + OFF_K + 2 * BOX, &mR, rope_full, 0, j * BKV, b);
      }
      mbar_drain(q_full, 0);
      if (j < n_kv && j > 0) mbar_drain(rope_full, (j - 1) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait_or_abort(q_full, 0, abort_flag, 93);
      bool issued = false;
      int it = 0;
      const uint32_t q_base = smem_u32(smem + OFF_Q);
      const uint32_t k_base = smem_u32(smem + OFF_K);
      const uint32_t v_base = smem_u32(smem + OFF_V);
      auto rebuild = [&](int j) -> bool {  // Kacc = c_kv_j W_UK_h, Vacc = c_kv_j W_UV_h
        if (j > 0 && !mbar_wait_or_abort(acc_free, (j - 1) & 1, abort_flag, 94)) return false;
        tc_fence_after();
        for (int c = 0; c < NCHUNK; ++c, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_or_abort(&st_full[s], (it / STAGES) & 1, abort_flag, 95)) return false;
          tc_fence_after();
          const uint32_t a = smem_u32(smem + OFF_RING + s * CHUNK_BYTES);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = sdesc_sw128(a + k * 32, 16, 1024);
            mma_ss(tmem + COL_KA, ad, sdesc_sw128(a + BOX + k * 2048, WBOX, 1024), IDESC_RC, (c | k) ? 1u : 0u);
            mma_ss(tmem + COL_VA, ad, sdesc_sw128(a + BOX + 2 * WBOX + k * 2048, WBOX, 1024), IDESC_RC,
                   (c | k) ? 1u : 0u);
          }
          issued = true;
          mma_commit(&st_empty[s]);
        }
        mma_commit(acc_full);
        return true;
      };
      if (ok) ok = rebuild(0);
      for (int j = 0; j < n_kv && ok; ++j) {
        // S(j) = Q [K_nope | k_rope]^T once the convert warps wrote tile j
        if (!mbar_wait_or_abort(kt_full, j & 1, abort_flag, 96) ||
            !mbar_wait_or_abort(rope_full, j & 1, abort_flag, 97)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 12; ++kk) {
          const uint32_t c = kk >> 2, k = kk & 3;
          mma_ss(tmem + COL_S, sdesc_sw128(q_base + c * BOX + k * 32, 16, 1024),
                 sdesc_sw128(k_base + c * BOX + k * 32, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        if (j + 1 < n_kv && !rebuild(j + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait_or_abort(p_full, j & 1, abort_flag, 98)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          mma_ts(tmem + COL_O, tmem + COL_S + kk * 8, sdesc_sw128(v_base + kk * 2048, BOX, 1024), IDESC_PV,
                 (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(kv_free);
      }
      if (ok) {
        mma_commit(o_done);
      } else if (issued) {
        mma_commit(drain);
        mbar_drain(drain, 0);
      }
    }
  } else if (warp < 6) {
    // ---------------------------------------------- softmax: one query row per thread
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int q_row = t * BQ + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int limit = p.causal ? p.q_offset + q_row : p.S - 1;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      // s_full(j) also covers PV(j-1): O is stable when it fires
      if (!warp_wait(s_full, j & 1, 101)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = tmem + COL_S + lane_off;
      float x[128];
      {
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(s_addr + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(u[i]) * p.scale_log2;
        }
      }
      const int kv0 = j * BKV;
      if (kv0 + BKV - 1 > limit) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (kv0 + i > limit) x[i] = -INFINITY;
      }
      float mt = x[0];
#pragma unroll
      for (int i = 1; i < 128; ++i) mt = fmaxf(mt, x[i]);
      float m_use = m_run, alpha = 1.f;
      bool rescale = false;
      if (m_run == -INFINITY) {
        m_use = mt;
      } else if (mt > m_run + RESCALE_THRESHOLD) {
        m_use = mt;
        alpha = ex2_approx(m_run - mt);
        rescale = true;
      }
      const float m_sub = m_use == -INFINITY ? 0.f : m_use;
      float sum = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float p0 = ex2_approx(x[2 * i] - m_sub);
        const float p1 = ex2_approx(x[2 * i + 1] - m_sub);
        sum += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + sum;
      m_run = m_use;
      {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = pk[c * 32 + i];
          tmem_st32(s_addr + c * 32, w);
        }
      }
      if (__any_sync(0xffffffffu, rescale)) {
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
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && warp_wait(o_done, 0, 102)) {
      tc_fence_after();
      const uint32_t o_addr = tmem + COL_O + lane_off;
      const bool valid = q_row < p.Sq;
      const float inv = 1.f / l_run;
      bf16* orow = p.out + ((static_cast<long long>(b) * p.Sq + q_row) * p.n_h + h) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
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
      if (valid)
        p.lse[(static_cast<long long>(b) * p.n_h + h) * p.Sq + q_row] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
    }
  } else {
    // ---------------------------------------------- convert: Kacc / Vacc -> bf16 operand tiles
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    for (int j = 0; j < n_kv; ++j) {
      if (!warp_wait(acc_full, j & 1, 111)) break;
      if (j > 0 && !warp_wait(kv_free, (j - 1) & 1, 112)) break;  // S(j-1), PV(j-1) done reading
      tc_fence_after();
#pragma unroll 1
      for (int m = 0; m < 2; ++m) {  // m = 0: K_nope tile, m = 1: V tile
        const uint32_t acc = tmem + (m == 0 ? COL_KA : COL_VA) + lane_off;
        uint8_t* tile = smem + (m == 0 ? OFF_K : OFF_V);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {  // 32 columns = 4 chunks of 16 bytes in box c / 2
          uint32_t u[32];
          tmem_ld32(acc + c * 32, u);
          tmem_wait_ld();
          uint8_t* box = tile + (c >> 1) * BOX;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(u[8 * q + 0]), __uint_as_float(u[8 * q + 1]));
            w.y = pack_bf16x2(__uint_as_float(u[8 * q + 2]), __uint_as_float(u[8 * q + 3]));
            w.z = pack_bf16x2(__uint_as_float(u[8 * q + 4]), __uint_as_float(u[8 * q + 5]));
            w.w = pack_bf16x2(__uint_as_float(u[8 * q + 6]), __uint_as_float(u[8 * q + 7]));
            *reinterpret_cast<uint4*>(box + sw128_offset(r, (c & 1) * 4 + q)) = w;
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(acc_free);
        mbar_arrive(kt_full);
      }
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

LaunchResult tc_attn_fwd_fused(const Dims& d, const bf16* q, const bf16* c_kv, const bf16* W_UK, const bf16* W_UV,
                               const bf16* k_rope, bf16* out, float* lse, cudaStream_t st) {
  LaunchResult r;
  CUtensorMap mQ, mC, mWK, mWV, mR;
  {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 192;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    const uint32_t box[3] = {64, BQ, 1};
    r.cu = make_tmap(&mQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[3] = {static_cast<uint64_t>(d.d_c), static_cast<uint64_t>(d.S), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {static_cast<uint64_t>(d.d_c) * 2, static_cast<uint64_t>(d.S) * d.d_c * 2};
    const uint32_t box[3] = {64, BKV, 1};
    r.cu = make_tmap(&mC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c_kv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t n = static_cast<uint64_t>(d.n_h) * 128;
    const uint64_t dims[2] = {n, static_cast<uint64_t>(d.d_c)};
    const uint64_t strides[1] = {n * 2};
    const uint32_t box[2] = {64, 64};
    r.cu = make_tmap(&mWK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W_UK, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r.cu == CUDA_SUCCESS)
      r.cu = make_tmap(&mWV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W_UV, dims, strides, box,
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
    r.what = "tensor maps fused-reconstruction forward";
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
  p.scale_log2 = d.scale * LOG2E;
  p.out = out;
  p.lse = lse;
  r.err = cudaFuncSetAttribute(attn_fwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(attn_fwd_fused)";
    return r;
  }
  attn_fwd_fused_kernel<<<dim3(p.n_q_tiles, d.n_h, d.B), NTHREADS, SMEM_BYTES, st>>>(mQ, mC, mWK, mWV, mR, p);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "attn_fwd_fused_kernel launch";
  return r;
}

}  // namespace laga
