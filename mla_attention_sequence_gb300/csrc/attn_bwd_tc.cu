// Causal attention backward on the tensor cores for the LAGA MLA block
// (d_qk = 128 + 64, d_v = 128, bf16 operands, fp32 accumulation).
//
// One CTA per (128-row key tile, head, batch element); it walks the 64-row
// query tiles that can see its keys. Everything is computed transposed (keys
// on the TMEM lanes), from the closed-form softmax gradient:
//   S^T  = K Q^T                 P^T  = exp(S^T * scale - lse)
//   dP^T = V dO^T                dS^T = P^T o (dP^T - D)
//   dV  += P^T dO                dK  += dS^T Q      (scale applied at the end)
//   dQ^T = K^T dS^T              added to an fp32 dq accumulator with red.add
// dV, dK_nope and this head's RoPE-key gradient stay in TMEM for the whole
// walk and are written once at the end.
//
// Warp roles (320 threads):
//   warp 0      lane 0: TMA for the key/value tile once, then Q, dO, lse, D tiles
//   warp 1      TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 2..5  "softmax": one key row per thread; P^T and dS^T to shared memory
//   warps 6..9  "drain": dQ^T rows (one head dim per thread) to the accumulator
// TMEM columns: dV [0,128), dK_nope [128,256), dK_rope [256,320), and three
// 64-column regions [320,512) that rotate between S^T, dP^T and the two
// halves of dQ^T, so S^T of the next query tile can be computed while dQ^T of
// the current one drains.
#include "internal.h"
#include "ptx.cuh"

namespace laga {
namespace {

constexpr int BKV = 128;
constexpr int BQ = 64;
constexpr int KBOX = 16384;  // [128 rows][64] bf16
constexpr int QBOX = 8192;   // [64 rows][64] bf16
constexpr int K_BYTES = 3 * KBOX;
constexpr int V_BYTES = 2 * KBOX;
constexpr int Q_BYTES = 3 * QBOX;
constexpr int DO_BYTES = 2 * QBOX;
constexpr int ROWV_BYTES = BQ * 4;  // lse or D for one query tile
constexpr int STAGE_BYTES = Q_BYTES + DO_BYTES;
constexpr int PT_BYTES = BKV * BQ * 2;  // [128 keys][64 queries] bf16
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + K_BYTES;
constexpr int OFF_STAGE = OFF_V + V_BYTES;
constexpr int OFF_PT = OFF_STAGE + 2 * STAGE_BYTES;
constexpr int OFF_DS = OFF_PT + 2 * PT_BYTES;
constexpr int OFF_ROWV = OFF_DS + 2 * PT_BYTES;
constexpr int OFF_BARS = OFF_ROWV + 2 * 2 * ROWV_BYTES;
constexpr int SMEM_BYTES = OFF_BARS + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_DV = 0, COL_DKN = 128, COL_DKR = 256, COL_R0 = 320;
constexpr uint32_t IDESC_N64_KK = idesc_bf16(128, 64, false, false);   // S^T, dP^T
constexpr uint32_t IDESC_N128_KM = idesc_bf16(128, 128, false, true);  // dV, dK_nope
constexpr uint32_t IDESC_N64_KM = idesc_bf16(128, 64, false, true);    // dK_rope
constexpr uint32_t IDESC_N64_MM = idesc_bf16(128, 64, true, true);     // dQ^T
constexpr int NTHREADS = 320;

struct BwdParams {
  int* status;  // device status word (timeouts)
  int Sq, S, n_h, q_offset, causal, skv_pad, sq_pad;
  float scale;       // softmax scale (dK is scaled once at the end)
  float scale_log2;  // scale * log2(e)
  const float* lse2;
  const float* delta;
  float* dq_acc;
  bf16* dk_ws;
  bf16* dv_ws;
  float* dkr_ws;
};

// Region holding S^T (and later dQ^T_a) / dP^T (later dQ^T_b) for query step i.
__device__ __forceinline__ uint32_t region_a(int i) { return COL_R0 + 64u * ((3 - i % 3) % 3); }
__device__ __forceinline__ uint32_t region_b(int i) { return COL_R0 + 64u * ((4 - i % 3) % 3); }

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mR, const __grid_constant__ CUtensorMap mV,
                    const __grid_constant__ CUtensorMap mdO, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;      // [2]
  uint64_t* q_empty = bars + 3;     // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* dp_full = bars + 6;
  uint64_t* pt_full = bars + 7;
  uint64_t* ds_full = bars + 8;
  uint64_t* smem_free = bars + 9;   // [2]
  uint64_t* dq_full = bars + 11;
  uint64_t* rfree_a = bars + 12;
  uint64_t* rfree_b = bars + 13;
  uint64_t* acc_done = bars + 14;
  uint64_t* drain = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x;  // key tile: lower tiles see more queries, so launch them first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kv0 = n * BKV;
  const int first_qt = p.causal ? max(0, kv0 - p.q_offset) / BQ : 0;
  const int n_qt = (p.Sq + BQ - 1) / BQ - first_qt;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&smem_free[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(pt_full, 4);
    mbar_init(ds_full, 4);
    mbar_init(dq_full, 1);
    mbar_init(rfree_a, 4);
    mbar_init(rfree_b, 4);
    mbar_init(acc_done, 1);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mR);
      tma_prefetch_desc(&mV);
      tma_prefetch_desc(&mdO);
      mbar_arrive_expect_tx(kv_full, K_BYTES + V_BYTES);
      const int krow = b * p.skv_pad + kv0;
      tma_load_2d(smem + OFF_K, &mK, kv_full, h * 128, krow);
      tma_load_2d(smem + OFF_K + KBOX, &mK, kv_full, h * 128 + 64, krow);
      tma_load_3d(smem + OFF_K + 2 * KBOX, &mR, kv_full, 0, kv0, b);
      tma_load_2d(smem + OFF_V, &mV, kv_full, h * 128, krow);
      tma_load_2d(smem + OFF_V + KBOX, &mV, kv_full, h * 128 + 64, krow);
      int i = 0;
      for (; i < n_qt; ++i) {
        const int s = i & 1;
        if (!mbar_wait_or_abort(&q_empty[s], ((i >> 1) & 1) ^ 1, abort_flag, 21)) break;
        const int q0 = (first_qt + i) * BQ;
        uint8_t* st = smem + OFF_STAGE + s * STAGE_BYTES;
        float* rows = reinterpret_cast<float*>(smem + OFF_ROWV) + s * 2 * BQ;
        mbar_arrive_expect_tx(&q_full[s], STAGE_BYTES + 2 * ROWV_BYTES);
        tma_load_3d(st, &mQ, &q_full[s], h * 192, q0, b);
        tma_load_3d(st + QBOX, &mQ, &q_full[s], h * 192 + 64, q0, b);
        tma_load_3d(st + 2 * QBOX, &mQ, &q_full[s], h * 192 + 128, q0, b);
        tma_load_3d(st + Q_BYTES, &mdO, &q_full[s], h * 128, q0, b);
        tma_load_3d(st + Q_BYTES + QBOX, &mdO, &q_full[s], h * 128 + 64, q0, b);
        const long long roff = (static_cast<long long>(b) * p.n_h + h) * p.sq_pad + q0;
        bulk_load(rows, p.lse2 + roff, ROWV_BYTES, &q_full[s]);
        bulk_load(rows + BQ, p.delta + roff, ROWV_BYTES, &q_full[s]);
      }
      if (i < n_qt) {
        mbar_drain(kv_full, 0);
        for (int k = i - 2 < 0 ? 0 : i - 2; k < i; ++k) mbar_drain(&q_full[k & 1], (k >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait_or_abort(kv_full, 0, abort_flag, 22);
      bool issued = false;
      tc_fence_after();
      const uint32_t k_base = smem_u32(smem + OFF_K);
      const uint32_t v_base = smem_u32(smem + OFF_V);
      for (int i = 0; i < n_qt && ok; ++i) {
        const int s = i & 1;
        const uint32_t ra = tmem + region_a(i), rb = tmem + region_b(i);
        if (!mbar_wait_or_abort(&q_full[s], (i >> 1) & 1, abort_flag, 23)) { ok = false; break; }
        if (i >= 2 && !mbar_wait_or_abort(rfree_b, (i - 2) & 1, abort_flag, 24)) { ok = false; break; }
        tc_fence_after();
        const uint32_t q_base = smem_u32(smem + OFF_STAGE + s * STAGE_BYTES);
        const uint32_t do_base = q_base + Q_BYTES;
        // S^T = K Q^T   (K-dim 192: two no-RoPE boxes and the RoPE box)
#pragma unroll
        for (int kk = 0; kk < 12; ++kk) {
          const uint32_t c = kk >> 2, k = kk & 3;
          mma_ss(ra, sdesc_sw128(k_base + c * KBOX + k * 32, 16, 1024),
                 sdesc_sw128(q_base + c * QBOX + k * 32, 16, 1024), IDESC_N64_KK, kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        issued = true;
        if (i >= 1 && !mbar_wait_or_abort(rfree_a, (i - 1) & 1, abort_flag, 25)) { ok = false; break; }
        tc_fence_after();
        // dP^T = V dO^T  (K-dim 128)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t c = kk >> 2, k = kk & 3;
          mma_ss(rb, sdesc_sw128(v_base + c * KBOX + k * 32, 16, 1024),
                 sdesc_sw128(do_base + c * QBOX + k * 32, 16, 1024), IDESC_N64_KK, kk > 0 ? 1u : 0u);
        }
        mma_commit(dp_full);
        const uint32_t pt_base = smem_u32(smem + OFF_PT + s * PT_BYTES);
        const uint32_t ds_base = smem_u32(smem + OFF_DS + s * PT_BYTES);
        if (!mbar_wait_or_abort(pt_full, i & 1, abort_flag, 26)) { ok = false; break; }
        tc_fence_after();
        // dV += P^T dO   (K-dim = 64 queries; dO read MN-major)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem + COL_DV, sdesc_sw128(pt_base + k * 32, 16, 1024),
                 sdesc_sw128(do_base + k * 2048, QBOX, 1024), IDESC_N128_KM, (i > 0 || k > 0) ? 1u : 0u);
        if (!mbar_wait_or_abort(ds_full, i & 1, abort_flag, 27)) { ok = false; break; }
        tc_fence_after();
        // dK_nope += dS^T Q_nope ; dK_rope += dS^T Q_rope
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t a = sdesc_sw128(ds_base + k * 32, 16, 1024);
          mma_ss(tmem + COL_DKN, a, sdesc_sw128(q_base + k * 2048, QBOX, 1024), IDESC_N128_KM,
                 (i > 0 || k > 0) ? 1u : 0u);
          mma_ss(tmem + COL_DKR, a, sdesc_sw128(q_base + 2 * QBOX + k * 2048, QBOX, 1024), IDESC_N64_KM,
                 (i > 0 || k > 0) ? 1u : 0u);
        }
        // dQ^T = K^T dS^T: head dims [0,128) into region a, [64,192) into region b
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bd = sdesc_sw128(ds_base + k * 2048, KBOX, 1024);
          mma_ss(ra, sdesc_sw128(k_base + k * 2048, KBOX, 1024), bd, IDESC_N64_MM, k > 0 ? 1u : 0u);
          mma_ss(rb, sdesc_sw128(k_base + KBOX + k * 2048, KBOX, 1024), bd, IDESC_N64_MM, k > 0 ? 1u : 0u);
        }
        mma_commit(dq_full);
        mma_commit(&smem_free[s]);
        mma_commit(&q_empty[s]);
      }
      if (ok) {
        mma_commit(acc_done);
      } else if (issued) {
        mma_commit(drain);
        mbar_drain(drain, 0);
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row within the tile
    const int kv = kv0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
      return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    };
    for (int i = 0; i < n_qt; ++i) {
      const int s = i & 1;
      const int q0 = (first_qt + i) * BQ;
      if (i >= 2 && !warp_wait(&smem_free[s], ((i >> 1) - 1) & 1, 31)) { ok = false; break; }
      if (!warp_wait(&q_full[s], (i >> 1) & 1, 32)) { ok = false; break; }
      if (!warp_wait(s_full, i & 1, 33)) { ok = false; break; }
      tc_fence_after();
      const float* rows = reinterpret_cast<const float*>(smem + OFF_ROWV) + s * 2 * BQ;
      const int limit = p.causal ? kv - p.q_offset : (kv < p.S ? p.Sq : -1);  // queries i >= limit see key kv
      float pr[64];
      {
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld32(tmem + region_a(i) + lane_off + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int qi = c * 32 + k;
            const bool vis = p.causal ? (q0 + qi >= limit) : (limit > 0);
            const float x = fmaf(__uint_as_float(u[k]), p.scale_log2, -rows[qi]);
            pr[qi] = vis ? ex2_approx(x) : 0.f;
          }
        }
      }
      uint8_t* pt = smem + OFF_PT + s * PT_BYTES;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 w;
        w.x = pack_bf16x2(pr[8 * c + 0], pr[8 * c + 1]);
        w.y = pack_bf16x2(pr[8 * c + 2], pr[8 * c + 3]);
        w.z = pack_bf16x2(pr[8 * c + 4], pr[8 * c + 5]);
        w.w = pack_bf16x2(pr[8 * c + 6], pr[8 * c + 7]);
        *reinterpret_cast<uint4*>(pt + sw128_offset(r, c)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pt_full);
      if (!warp_wait(dp_full, i & 1, 34)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld32(tmem + region_b(i) + lane_off + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int qi = c * 32 + k;
            pr[qi] = pr[qi] * (__uint_as_float(u[k]) - rows[BQ + qi]);
          }
        }
      }
      uint8_t* ds = smem + OFF_DS + s * PT_BYTES;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 w;
        w.x = pack_bf16x2(pr[8 * c + 0], pr[8 * c + 1]);
        w.y = pack_bf16x2(pr[8 * c + 2], pr[8 * c + 3]);
        w.z = pack_bf16x2(pr[8 * c + 4], pr[8 * c + 5]);
        w.w = pack_bf16x2(pr[8 * c + 6], pr[8 * c + 7]);
        *reinterpret_cast<uint4*>(ds + sw128_offset(r, c)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    // epilogue: dV (bf16) and this head's RoPE-key gradient (fp32), scaled
    if (ok && warp_wait(acc_done, 0, 35)) {
      tc_fence_after();
      const long long row = static_cast<long long>(b) * p.skv_pad + kv;
      bf16* dv = p.dv_ws + row * (static_cast<long long>(p.n_h) * 128) + h * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + COL_DV + lane_off + c * 32, u);
        tmem_wait_ld();
        uint4* dst = reinterpret_cast<uint4*>(dv + c * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(u[8 * v + 0]), __uint_as_float(u[8 * v + 1]));
          w.y = pack_bf16x2(__uint_as_float(u[8 * v + 2]), __uint_as_float(u[8 * v + 3]));
          w.z = pack_bf16x2(__uint_as_float(u[8 * v + 4]), __uint_as_float(u[8 * v + 5]));
          w.w = pack_bf16x2(__uint_as_float(u[8 * v + 6]), __uint_as_float(u[8 * v + 7]));
          dst[v] = w;
        }
      }
      float* dkr = p.dkr_ws + (row * p.n_h + h) * 64;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + COL_DKR + lane_off + c * 32, u);
        tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(dkr + c * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          dst[v] = make_float4(__uint_as_float(u[4 * v]) * p.scale, __uint_as_float(u[4 * v + 1]) * p.scale,
                               __uint_as_float(u[4 * v + 2]) * p.scale, __uint_as_float(u[4 * v + 3]) * p.scale);
      }
    }
  } else {
    // ------------------------------------------------------------ drain warps
    const int quarter = warp & 3;
    const int dlane = quarter * 32 + lane;  // TMEM lane = head dim row of dQ^T
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
      return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    };
    const long long q_stride = static_cast<long long>(p.n_h) * 192;
    for (int i = 0; i < n_qt; ++i) {
      const int q0 = (first_qt + i) * BQ;
      if (!warp_wait(dq_full, i & 1, 41)) { ok = false; break; }
      tc_fence_after();
      float* base = p.dq_acc + (static_cast<long long>(b) * p.Sq + q0) * q_stride + h * 192;
      const int nq = min(BQ, p.Sq - q0);
      {
        uint32_t ua[32], ub[32];
        tmem_ld32(tmem + region_a(i) + lane_off, ua);
        tmem_ld32(tmem + region_a(i) + lane_off + 32, ub);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(rfree_a);
        float* col = base + dlane;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k < nq) atomicAdd(col + k * q_stride, __uint_as_float(ua[k]));
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (32 + k < nq) atomicAdd(col + (32 + k) * q_stride, __uint_as_float(ub[k]));
      }
      if (quarter >= 2) {
        uint32_t ua[32], ub[32];
        tmem_ld32(tmem + region_b(i) + lane_off, ua);
        tmem_ld32(tmem + region_b(i) + lane_off + 32, ub);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(rfree_b);
        float* col = base + 64 + dlane;  // lane 64 + x holds head dim 128 + x
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k < nq) atomicAdd(col + k * q_stride, __uint_as_float(ua[k]));
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (32 + k < nq) atomicAdd(col + (32 + k) * q_stride, __uint_as_float(ub[k]));
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(rfree_b);
      }
    }
    // epilogue: dK_nope (scaled, bf16)
    if (ok && warp_wait(acc_done, 0, 42)) {
      tc_fence_after();
      const long long row = static_cast<long long>(b) * p.skv_pad + kv0 + dlane;
      bf16* dk = p.dk_ws + row * (static_cast<long long>(p.n_h) * 128) + h * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + COL_DKN + lane_off + c * 32, u);
        tmem_wait_ld();
        uint4* dst = reinterpret_cast<uint4*>(dk + c * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(u[8 * v + 0]) * p.scale, __uint_as_float(u[8 * v + 1]) * p.scale);
          w.y = pack_bf16x2(__uint_as_float(u[8 * v + 2]) * p.scale, __uint_as_float(u[8 * v + 3]) * p.scale);
          w.z = pack_bf16x2(__uint_as_float(u[8 * v + 4]) * p.scale, __uint_as_float(u[8 * v + 5]) * p.scale);
          w.w = pack_bf16x2(__uint_as_float(u[8 * v + 6]) * p.scale, __uint_as_float(u[8 * v + 7]) * p.scale);
          dst[v] = w;
        }
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

LaunchResult tc_attn_bwd(const Dims& d, const bf16* q, const bf16* k_rope, const bf16* dout, const BwdWorkspace& w,
                         cudaStream_t st) {
  LaunchResult r;
  CUtensorMap mQ, mK, mR, mV, mdO;
  {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 192;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    const uint32_t box[3] = {64, 64, 1};
    r.cu = make_tmap(&mQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t inner = static_cast<uint64_t>(d.n_h) * 128;
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(d.Sq), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {inner * 2, inner * 2 * d.Sq};
    const uint32_t box[3] = {64, 64, 1};
    r.cu = make_tmap(&mdO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dout, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t kv_inner = static_cast<uint64_t>(d.n_h) * 128;
  const uint64_t kv_rows = static_cast<uint64_t>(d.B) * d.skv_pad;
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[2] = {kv_inner, kv_rows};
    const uint64_t strides[1] = {kv_inner * 2};
    const uint32_t box[2] = {64, 128};
    r.cu = make_tmap(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.k_ws, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    if (r.cu == CUDA_SUCCESS)
      r.cu = make_tmap(&mV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.v_ws, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(d.S), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(d.S) * 128};
    const uint32_t box[3] = {64, 128, 1};
    r.cu = make_tmap(&mR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_rope, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps attention backward";
    return r;
  }
  BwdParams p{};
  p.Sq = d.Sq;
  p.S = d.S;
  p.n_h = d.n_h;
  p.q_offset = d.q_offset;
  p.causal = d.causal ? 1 : 0;
  p.skv_pad = d.skv_pad;
  p.sq_pad = d.sq_pad;
  p.scale = d.scale;
  p.scale_log2 = d.scale * 1.4426950408889634f;
  p.lse2 = w.lse2;
  p.delta = w.delta;
  p.dq_acc = w.dq_acc;
  p.dk_ws = w.dk_ws;
  p.dv_ws = w.dv_ws;
  p.dkr_ws = w.dkr_ws;
  p.status = device_status_ptr();
  r.err = cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(attn_bwd)";
    return r;
  }
  attn_bwd_kernel<<<dim3(d.skv_pad / BKV, d.n_h, d.B), NTHREADS, SMEM_BYTES, st>>>(mQ, mK, mR, mV, mdO, p);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "attn_bwd_kernel launch";
  return r;
}

}  // namespace laga
