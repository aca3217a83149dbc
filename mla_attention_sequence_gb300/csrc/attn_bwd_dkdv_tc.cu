// Attention backward, key/value side: dV, dK_nope and each head's RoPE-key
// gradient, on the tensor cores (d_qk = 128 + 64, d_v = 128, bf16 operands,
// fp32 accumulation).
//
// One CTA per (128-row key tile, group of G consecutive heads, batch element);
// for each head of its group in turn it walks the 64-row query tiles that can
// see its keys. Keys sit on the TMEM lanes:
//   S^T  = K Q^T          P^T  = exp(S^T * scale - lse)
//   dP^T = V dO^T         dS^T = P^T o (dP^T - D)
//   dV  += P^T dO         dK  += dS^T Q        (scale applied once at the end)
// P^T and dS^T are written back into TMEM as packed bf16 over S^T / dP^T and
// feed the dV / dK products as the A operand straight from TMEM, so they never
// touch shared memory. dK covers all 192 head dims in one N = 192 product: the
// first 128 columns are dK_nope, the last 64 the RoPE-key gradient, which is one
// tensor shared by every head: those columns keep accumulating over the group's
// G heads and are written once per CTA (fp32, one partial per head group).
//
// Head boundaries. A CTA pays its start (TMEM, barriers, the first tiles' load
// latency) once for G heads. When head u's last dP^T has been issued, the MMA
// warp releases the key/value tile (kv_empty) and the producer loads head u+1's
// K_nope and V over it (the RoPE key stays). The key-row warps move dV to global
// memory as soon as head u's last dV has finished (dv_done), while the tensor
// pipe still runs its last dK; when that has finished (acc_done) they move
// dK_nope, zero its columns and release the accumulators (acc_free) for head
// u+1's first dV, while the tensor pipe already runs head u+1's first S^T and dP^T.
//
// Warp roles (352 threads):
//   warp 0      lane 0: TMA for the key/value tile, then Q, dO, lse, D tiles
//   warp 1      TMEM allocation; issues every tcgen05.mma and touches no shared
//               memory in its loop: it learns that an operand is ready from
//   warp 10     the waiter, which waits on each mbarrier the next MMA group needs
//               and meets warp 1 at a named barrier (the AND of their flags
//               carries a timeout). Measured on GB300: an mbarrier test in the
//               MMA warp costs the tensor pipe 150-400 cycles per step once
//               compute warps share its SM sub-partition; the named barrier
//               costs it next to nothing.
//   warps 2..9  two warpgroups; each thread owns one key row (TMEM lane) and
//               half of the 64 query columns: P^T, dS^T, and half of each
//               head's accumulator drain
// TMEM columns: dV [0,128), dK [128,320), S^T x2 [320,448), dP^T [448,512).
// Step i packs P^T(i) AND dS^T(i) into its own S^T buffer (P^T over the first
// 16 of each warpgroup's 32 score columns, dS^T over the other 16), so the dP^T
// columns are free as soon as the softmax has read dP^T(i) into registers.
// MMA order S(0) dP(0) S(1) | dV(i) dP(i+1) dK(i) S(i+2) | ...: dP(i+1) no longer
// waits behind dK(i), which leaves every hand-off (P^T, dP^T read, dS^T) most of
// a step of slack instead of a few hundred cycles (measured on GB300: with the
// order dV(i) dK(i) dP(i+1) S(i+2) and dS^T over dP^T, the MMA warp waited
// ~400 cycles per step at the P^T and dS^T hand-offs, 1820 cycles per step
// against 1600 of tensor work).
#include "internal.h"
#include "ptx.cuh"

LAGA_TRACE_DEFINE(dkdv)

namespace laga {
namespace {

constexpr int BKV = 128;
constexpr int BQ = 64;
constexpr int NSTAGE = 3;
constexpr int KBOX = 16384;  // [128 rows][64] bf16
constexpr int QBOX = 8192;   // [64 rows][64] bf16
constexpr int K_BYTES = 3 * KBOX;
constexpr int V_BYTES = 2 * KBOX;
constexpr int Q_BYTES = 3 * QBOX;
constexpr int DO_BYTES = 2 * QBOX;
constexpr int ROWV_BYTES = BQ * 4;
constexpr int STAGE_BYTES = Q_BYTES + DO_BYTES;  // 40 KB, 1024-aligned
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + K_BYTES;
constexpr int OFF_STAGE = OFF_V + V_BYTES;
constexpr int OFF_ROWV = OFF_STAGE + NSTAGE * STAGE_BYTES;
// per key-row warp, a [32 rows][64 B] scratch (64-byte swizzle, 512-byte aligned)
// from which the accumulator drain's tensor-map stores read
constexpr int SCR_BYTES = 32 * 64;
constexpr int OFF_SCR = OFF_ROWV + NSTAGE * 2 * ROWV_BYTES;
constexpr int OFF_BARS = OFF_SCR + 8 * SCR_BYTES;
constexpr int SMEM_BYTES = OFF_BARS + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_S = 320, COL_DP = 448;
constexpr uint32_t IDESC_ST = idesc_bf16(128, 64, false, false);   // S^T, dP^T
constexpr uint32_t IDESC_DV = idesc_bf16(128, 128, false, true);   // dV (A from TMEM)
constexpr uint32_t IDESC_DK = idesc_bf16(128, 192, false, true);   // dK (A from TMEM)
constexpr int NTHREADS = 352;
constexpr int WAITER_WARP = 10;
constexpr int HANDOFF_BAR = 1;  // named barrier of warp 1 and the waiter (64 threads)
constexpr uint32_t SOFTMAX_WARPS = 8;

// TMEM column (within a step's S^T buffer) of packed bf16 chunk k (16 queries)
// of P^T: the two warpgroups pack their halves at [0,16) and [32,48); of dS^T:
// at [16,32) and [48,64), the score columns each warpgroup has read already.
__device__ __forceinline__ uint32_t packed_col(int k) { return 8u * k + 16u * (k >> 1); }
__device__ __forceinline__ uint32_t packed_col_ds(int k) { return 16u + 8u * k + 16u * (k >> 1); }

struct Params {
  int* status;
  int Sq, S, n_h, q_offset, causal, skv_pad, sq_pad;
  int G;     // heads per CTA (consecutive heads blockIdx.y * G ..)
  int n_hg;  // head groups = n_h / G: the RoPE-key partials per key row
  int q_split, q_offset2;  // second query segment (q_split = 0: none)
  int successor;  // linear block distance to the CTA that will next run on this SM (the SM count)
  float scale, scale_log2;
  const float* lse2;
  const float* delta;
};

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                         const __grid_constant__ CUtensorMap mR, const __grid_constant__ CUtensorMap mV,
                         const __grid_constant__ CUtensorMap mdO, const __grid_constant__ CUtensorMap mdK,
                         const __grid_constant__ CUtensorMap mdV, const __grid_constant__ CUtensorMap mdKR,
                         const Params p) {
  extern __shared__ uint8_t smem_raw[];
  LAGA_TRACE_CTA_BEGIN(dkdv);
  LAGA_TRACE_POINT(dkdv, 30, 0);
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;   // [NSTAGE]
  uint64_t* q_empty = bars + 4;  // [NSTAGE]
  uint64_t* s_full = bars + 7;   // [2]
  uint64_t* dp_full = bars + 9;
  // P^T of step i+1 can be ready before the MMA thread has seen step i's, so
  // p_full alternates between two barriers (one phase of each per two steps).
  uint64_t* p_full = bars + 10;  // [2]
  // dS^T(i) can complete before the waiter has seen dS^T(i-1) (dP(i) is issued
  // before that hand-off), so ds_full alternates between two barriers too.
  auto ds_full = [bars](int i) { return (i & 1) ? bars + 17 : bars + 12; };
  uint64_t* acc_done = bars + 13;  // a head's last dK is done (one phase per head)
  uint64_t* drain = bars + 14;
  uint64_t* dp_free = bars + 16;   // dP^T(i) read into registers: dP(i+1) may overwrite it
  uint64_t* kv_empty = bars + 18;  // a head's last dP^T is done: the next head's K_nope, V may load
  uint64_t* acc_free = bars + 19;  // dV and dK_nope drained (and dK_nope zeroed) for the next head
  uint64_t* dv_done = bars + 20;   // a head's last dV is done (one phase per head)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 25);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kv0 = blockIdx.x * BKV;  // low key tiles see the most queries: launched first
  const int hg = blockIdx.y;         // head group: heads hg * G .. hg * G + G - 1
  const int G = p.G;
  const int b = blockIdx.z;
  // The query tiles that see this key tile: a suffix of each segment's tiles,
  // walked segment 0 first. Step i of the walk is query tile qtile(i).
  const int nq = (p.Sq + BQ - 1) / BQ;
  const int seg_tiles = p.q_split > 0 ? p.q_split / BQ : nq;  // tiles of the first segment
  const int first0 = p.causal ? min(seg_tiles, max(0, kv0 - p.q_offset) / BQ) : 0;
  const int first1 = p.q_split > 0 ? seg_tiles + (p.causal ? min(nq - seg_tiles, max(0, kv0 - p.q_offset2) / BQ) : 0)
                                   : nq;
  const int n0 = seg_tiles - first0;
  const int n_qt = n0 + (nq - first1);
  auto qtile = [&](int i) { return i < n0 ? first0 + i : first1 + (i - n0); };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(&p_full[0], SOFTMAX_WARPS);
    mbar_init(&p_full[1], SOFTMAX_WARPS);
    mbar_init(ds_full(0), SOFTMAX_WARPS);
    mbar_init(ds_full(1), SOFTMAX_WARPS);
    mbar_init(dp_free, SOFTMAX_WARPS);
    mbar_init(acc_done, 1);
    mbar_init(dv_done, 1);
    mbar_init(drain, 1);
    mbar_init(kv_empty, 1);
    mbar_init(acc_free, SOFTMAX_WARPS);
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
      // Issue order: what the first MMAs need (the key/value tile, then the first
      // query stages), and only then L2 prefetches. Each TMA instruction takes the
      // issuing thread a while, and S(0) waits on all of the ones ahead of its tiles.
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mdO);
      const int krow = b * p.skv_pad + kv0;
      // Warm L2 with the first tiles of the CTA that will run next on this SM
      // (about one CTA lifetime from now): its start then waits on L2, not HBM.
      auto prefetch_successor = [&]() {
        const long long nx = gridDim.x, ny = gridDim.y;
        const long long nb = blockIdx.x + nx * (blockIdx.y + ny * blockIdx.z) + p.successor;
        if (nb < nx * ny * gridDim.z) {
          const int nkv0 = static_cast<int>(nb % nx) * BKV;
          const int nh = static_cast<int>((nb / nx) % ny) * G;
          const int nbb = static_cast<int>(nb / (nx * ny));
          const int nrow = nbb * p.skv_pad + nkv0;
          tma_prefetch_2d(&mK, nh * 128, nrow);
          tma_prefetch_2d(&mK, nh * 128 + 64, nrow);
          tma_prefetch_3d(&mR, 0, nkv0, nbb);
          tma_prefetch_2d(&mV, nh * 128, nrow);
          tma_prefetch_2d(&mV, nh * 128 + 64, nrow);
          const int nfirst = p.causal ? max(0, nkv0 - p.q_offset) / BQ : 0;
          for (int k = nfirst; k < nfirst + 2 && k < nq; ++k) {
            tma_prefetch_3d(&mQ, nh * 192, k * BQ, nbb);
            tma_prefetch_3d(&mQ, nh * 192 + 64, k * BQ, nbb);
            tma_prefetch_3d(&mQ, nh * 192 + 128, k * BQ, nbb);
            tma_prefetch_3d(&mdO, nh * 128, k * BQ, nbb);
            tma_prefetch_3d(&mdO, nh * 128 + 64, k * BQ, nbb);
          }
        }
      };
      bool ok = true;
      int gs = 0;  // global step: head u's step i is u * n_qt + i (stage ring, barrier phases)
      int kv_loads = 0;
      for (int u = 0; u < G && ok; ++u) {
        const int h = hg * G + u;
        if (u > 0 && !mbar_wait_or_abort(kv_empty, (u - 1) & 1, abort_flag, 57)) {
          ok = false;
          break;
        }
        // head u's K_nope and V over the previous head's; the RoPE key tile is shared
        mbar_arrive_expect_tx(kv_full, (u == 0 ? K_BYTES : 2 * KBOX) + V_BYTES);
        tma_load_2d(smem + OFF_K, &mK, kv_full, h * 128, krow);
        tma_load_2d(smem + OFF_K + KBOX, &mK, kv_full, h * 128 + 64, krow);
        if (u == 0) tma_load_3d(smem + OFF_K + 2 * KBOX, &mR, kv_full, 0, kv0, b);
        tma_load_2d(smem + OFF_V, &mV, kv_full, h * 128, krow);
        tma_load_2d(smem + OFF_V + KBOX, &mV, kv_full, h * 128 + 64, krow);
        ++kv_loads;
        for (int i = 0; i < n_qt; ++i, ++gs) {
          if (u + 1 < G && i == max(0, n_qt - 4)) {
            // the next head's key/value tile, into L2 a few steps before the boundary load
            tma_prefetch_2d(&mK, (h + 1) * 128, krow);
            tma_prefetch_2d(&mK, (h + 1) * 128 + 64, krow);
            tma_prefetch_2d(&mV, (h + 1) * 128, krow);
            tma_prefetch_2d(&mV, (h + 1) * 128 + 64, krow);
          }
          const int s = gs % NSTAGE;
          if (!mbar_wait_or_abort(&q_empty[s], ((gs / NSTAGE) & 1) ^ 1, abort_flag, 51)) {
            ok = false;
            break;
          }
          LAGA_TRACE_POINT(dkdv, 20, gs);
          const int q0 = qtile(i) * BQ;
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
          if (u == 0 && (i == NSTAGE - 1 || (i == n_qt - 1 && n_qt < NSTAGE))) prefetch_successor();
        }
      }
      if (n_qt <= 0) prefetch_successor();
      if (!ok) {
        // let copies already in flight land before shared memory goes away
        if (kv_loads > 0) mbar_drain(kv_full, (kv_loads - 1) & 1);
        for (int k = gs - NSTAGE < 0 ? 0 : gs - NSTAGE; k < gs; ++k)
          mbar_drain(&q_full[k % NSTAGE], (k / NSTAGE) & 1);
      }
    }
  } else if (warp == WAITER_WARP) {
    // The waiter walks the MMA warp's waits in the same order: per head u kv_full,
    // then per step (global index gs = u * n_qt + i) p_full(gs) (with, at a head's
    // first step after the first head, acc_free: the previous head's accumulators
    // drained), dp_free(gs) (i + 1 < n), ds_full(gs) (i >= 0) and q_full(gs+2)
    // (i + 2 < n). Each wait ends at the named barrier; a failed wait (timeout or
    // abort) is ANDed in, and both warps leave their loops at the same hand-off.
    auto handoff = [&](bool w) -> bool { return bar_and(HANDOFF_BAR, 64, w); };
    auto wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
      return warp_wait_or_abort(bar, parity, abort_flag, where);
    };
    bool all_ok = true;
    for (int u = 0; u < G && all_ok; ++u) {
      if (!handoff(wait(kv_full, u & 1, 52))) { all_ok = false; break; }
      for (int i = -2; i < n_qt; ++i) {
        const int gs = u * n_qt + i;
        if (i >= 0) {
          const bool freed = (i == 0 && u > 0) ? wait(acc_free, (u - 1) & 1, 58) : true;
          if (!handoff(freed && wait(&p_full[gs & 1], (gs >> 1) & 1, 54))) { all_ok = false; break; }
          if (i + 1 < n_qt && !handoff(wait(dp_free, gs & 1, 56))) { all_ok = false; break; }
          if (!handoff(wait(ds_full(gs), (gs >> 1) & 1, 55))) { all_ok = false; break; }
        }
        if (i + 2 < n_qt && !handoff(wait(&q_full[(gs + 2) % NSTAGE], ((gs + 2) / NSTAGE) & 1, 53))) {
          all_ok = false;
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // The whole warp runs the issue loop (an elected lane issues each block of MMAs).
    // Readiness comes from the waiter through the named barrier, never from a
    // shared-memory access of this warp.
    auto ready = [&]() -> bool {
      const bool r = bar_and(HANDOFF_BAR, 64, true);
      tc_fence_after();
      return r;
    };
    bool ok = true;
    bool issued = false;
    const uint64_t k_desc = sdesc_sw128(smem_u32(smem + OFF_K), 16, 1024);
    const uint64_t v_desc = sdesc_sw128(smem_u32(smem + OFF_V), 16, 1024);
    // K-major (16) and MN-major (QBOX) descriptors of a stage's Q and dO tiles
    auto stage_desc = [&](int i, uint32_t off, uint32_t lbo) {
      return sdesc_sw128(smem_u32(smem + OFF_STAGE + (i % NSTAGE) * STAGE_BYTES + off), lbo, 1024);
    };
    auto issue_s = [&](int i) {  // S^T(i) = K Q_i^T
      const uint64_t q_desc = stage_desc(i, 0, 16);
      const uint32_t d = tmem + COL_S + 64u * (i & 1);
#pragma unroll
      for (int c = 0; c < 3; ++c) {  // head dims [64c, 64c + 64): four K16 steps in box c
        const uint64_t a = k_desc + ((c * KBOX) >> 4), q = q_desc + ((c * QBOX) >> 4);
        mma4_ss_warp(d, a, a + 2, a + 4, a + 6, q, q + 2, q + 4, q + 6, IDESC_ST, c > 0 ? 1u : 0u);
      }
      mma_commit_warp(&s_full[i & 1]);
    };
    auto issue_dp = [&](int i) {  // dP^T(i) = V dO_i^T
      const uint64_t do_desc = stage_desc(i, Q_BYTES, 16);
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // value dims [64c, 64c + 64)
        const uint64_t a = v_desc + ((c * KBOX) >> 4), o = do_desc + ((c * QBOX) >> 4);
        mma4_ss_warp(tmem + COL_DP, a, a + 2, a + 4, a + 6, o, o + 2, o + 4, o + 6, IDESC_ST, c > 0 ? 1u : 0u);
      }
      mma_commit_warp(dp_full);
    };
    // One loop issues everything, the first steps included, so that every MMA
    // group exists once in the binary: code run once per CTA falls out of the
    // instruction cache between CTAs and then issues several times slower.
    // Per head u, iteration i: dV(i) (i >= 0); dP(i+1) (0 <= i+1 < n); dK(i)
    // (i >= 0); S(i+2) (i+2 < n). Steps are numbered globally (gs = u * n_qt + i)
    // for the stage ring, the S^T buffers and the barrier phases.
#ifdef LAGA_TRACE
    // trace build only: cycles spent at each hand-off
    long long st_cyc[3] = {0, 0, 0};
    const long long st_t0 = clock64();
#define DKDV_STAT_BEGIN(k) const long long w0_##k = clock64();
#define DKDV_STAT_END(k) st_cyc[k] += clock64() - w0_##k;
#else
#define DKDV_STAT_BEGIN(k)
#define DKDV_STAT_END(k)
#endif
    for (int u = 0; u < G && ok; ++u) {
      if (!ready()) { ok = false; break; }  // head u's key/value tile
      if (lane == 0) LAGA_TRACE_POINT(dkdv, 4, u);
      for (int i = -2; i < n_qt; ++i) {
        const int gs = u * n_qt + i;
        if (i >= 0) {
          DKDV_STAT_BEGIN(0)
          if (!ready()) { ok = false; break; }  // P^T(i) (and, at i = 0 after the first head, acc_free)
          DKDV_STAT_END(0)
          if (lane == 0) LAGA_TRACE_POINT(dkdv, 5, gs);
          // dV += P^T dO_i : A = P^T (TMEM, packed bf16), B = dO_i read MN-major
          const uint64_t do_mn = stage_desc(gs, Q_BYTES, QBOX);
          const uint32_t pt = tmem + COL_S + 64u * (gs & 1);
          mma4_ts_warp(tmem + COL_DV, pt + packed_col(0), pt + packed_col(1), pt + packed_col(2),
                       pt + packed_col(3), do_mn, do_mn + (2048 >> 4), do_mn + (4096 >> 4), do_mn + (6144 >> 4),
                       IDESC_DV, i > 0 ? 1u : 0u);
          if (i + 1 == n_qt) mma_commit_warp(dv_done);  // head u's dV is final
          if (i + 1 < n_qt) {
            if (!ready()) { ok = false; break; }  // dP^T(i) read out: dP(i+1) may overwrite it
            issue_dp(gs + 1);
            if (i + 2 == n_qt) mma_commit_warp(kv_empty);  // head u's last reader of K and V
          }
          DKDV_STAT_BEGIN(1)
          if (!ready()) { ok = false; break; }  // dS^T(i)
          DKDV_STAT_END(1)
          if (lane == 0) LAGA_TRACE_POINT(dkdv, 6, gs);
          // dK += dS^T Q_i : all 192 head dims in one product; dS^T(i) sits in S^T(i)'s
          // buffer. From the second head on dK_nope starts zeroed and the RoPE-key
          // columns carry the previous heads' sum, so every product accumulates.
          const uint64_t q_mn = stage_desc(gs, 0, QBOX);
          mma4_ts_warp(tmem + COL_DK, pt + packed_col_ds(0), pt + packed_col_ds(1), pt + packed_col_ds(2),
                       pt + packed_col_ds(3), q_mn, q_mn + (2048 >> 4), q_mn + (4096 >> 4), q_mn + (6144 >> 4),
                       IDESC_DK, (i > 0 || u > 0) ? 1u : 0u);
          mma_commit_warp(&q_empty[gs % NSTAGE]);
        } else if (i + 1 == 0 && n_qt > 0) {
          issue_dp(gs + 1);  // its stage was handed over before S(0)
          if (n_qt == 1) mma_commit_warp(kv_empty);
        }
        if (i + 2 < n_qt) {
          DKDV_STAT_BEGIN(2)
          if (!ready()) { ok = false; break; }  // Q_{i+2}, dO_{i+2}, lse and D rows
          DKDV_STAT_END(2)
          if (lane == 0) LAGA_TRACE_POINT(dkdv, 7, gs + 2);
          issue_s(gs + 2);
          issued = true;
          if (lane == 0) LAGA_TRACE_POINT(dkdv, 8, gs + 2);
        }
      }
      if (!ok) break;
      if (n_qt <= 0) {  // no MMA read the tile or wrote the accumulators
        mma_commit_warp(kv_empty);
        mma_commit_warp(dv_done);
      }
      mma_commit_warp(acc_done);  // head u's accumulators are final
    }
#ifdef LAGA_TRACE
    if (lane == 0) {
      for (int k = 0; k < 3; ++k) {
        LAGA_TRACE_STAT(dkdv, k, 0);
        LAGA_TRACE_STAT(dkdv, 3 + k, st_cyc[k]);
      }
      LAGA_TRACE_STAT(dkdv, 6, clock64() - st_t0);
      LAGA_TRACE_STAT(dkdv, 7, G * n_qt);
    }
#endif
#undef DKDV_STAT_BEGIN
#undef DKDV_STAT_END
    if (!ok && issued) {
      mma_commit_warp(drain);
      if (lane == 0) mbar_drain(drain, 0);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------ key-row warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // warpgroup: query columns [32*half, 32*half + 32)
    const int r = quarter * 32 + lane;
    const int kv = kv0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // local queries i >= q_min see this key (causal; per segment); non-causal: the key must exist
    const int q_min0 = p.causal ? kv - p.q_offset : (kv < p.S ? 0 : 0x7fffffff);
    const int q_min1 = p.causal ? kv - p.q_offset2 + p.q_split : q_min0;
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
      const bool all = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      __syncwarp();  // order lane 0's acquire before the other lanes' reads
      return all;
    };
    // Accumulator drain, straight from TMEM to global memory (the stage ring is busy
    // with the next head's tiles): warpgroup `half` moves dV and dK_nope columns
    // [64*half, 64*half + 64) of its 32 rows as bf16 (dK scaled by the softmax
    // scale) and, after the group's last head, the RoPE-key columns [32*half,
    // 32*half + 32) (fp32, this head group's partial). dV leaves once the head's
    // last dV has finished, while its last dK still runs; dK_nope once that has
    // finished, after which its columns are zeroed and both accumulators are
    // released (acc_free) for the next head's first dV and dK, while the tensor
    // pipe runs the next head's first S^T and dP^T. Both 32-column chunks of an
    // accumulator are loaded from TMEM together (one load latency per
    // accumulator); each chunk of the warp's 32 rows (64 bytes a row) then goes
    // registers -> the warp's scratch -> one tensor-map store, which the TMA unit
    // carries out while the warp goes on. (Global stores issued by the warp itself
    // held up its next shared-memory accesses, barrier waits included, until the
    // drain's 32 KB per warpgroup had left the SM: ~1K cycles before the next
    // head's first P^T could start.)
    uint8_t* scr = smem + OFF_SCR + (warp - 2) * SCR_BYTES;
    const int row0 = b * p.skv_pad + kv0 + quarter * 32;  // the warp's first row
    auto put_chunk = [&](const uint32_t (&w)[16], const CUtensorMap* map, int x) {
      if (lane == 0) bulk_wait_read_all();  // the previous chunk's store has read the scratch
      __syncwarp();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        *reinterpret_cast<uint4*>(scr + sw64_offset(lane, q4)) = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map, scr, x, row0);
        bulk_commit_group();
      }
    };
    const bool z = n_qt <= 0;  // no query sees this key tile: the accumulators were never written
    // this warpgroup's two 32-column chunks of dV (or dK_nope), both loads in flight
    auto drain_load = [&](bool is_dk, uint32_t (&a)[32], uint32_t (&c)[32]) {
      const uint32_t col = tmem + lane_off + (is_dk ? COL_DK : COL_DV) + 64 * half;
      tmem_ld32(col, a);
      tmem_ld32(col + 32, c);
    };
    // head hh's two loaded chunks, as bf16, to global memory
    auto drain_put = [&](int hh, bool is_dk, const uint32_t (&a)[32], const uint32_t (&c)[32]) {
      const float sc = is_dk ? p.scale : 1.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t(&v)[32] = j ? c : a;
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = z ? 0u : pack_bf16x2(__uint_as_float(v[2 * k]) * sc, __uint_as_float(v[2 * k + 1]) * sc);
        put_chunk(w, is_dk ? &mdK : &mdV, hh * 128 + 64 * half + 32 * j);
      }
    };
    auto release = [&](uint64_t* bar) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    for (int u = 0; u < G && ok; ++u) {
      const int h = hg * G + u;
      for (int i = 0; i < n_qt; ++i) {
        const int gs = u * n_qt + i;
        const int s = gs % NSTAGE;
        const int qt = qtile(i);
        const int qc = qt * BQ + 32 * half;  // this thread's first query column
        const int q_min = qt < seg_tiles ? q_min0 : q_min1;
        if (!warp_wait(&q_full[s], (gs / NSTAGE) & 1, 61)) { ok = false; break; }
        if (!warp_wait(&s_full[gs & 1], (gs >> 1) & 1, 62)) { ok = false; break; }
        if (lane == 0) LAGA_TRACE_POINT(dkdv, 10, gs);
        tc_fence_after();
        // this half-tile's 32 lse and D values (16-byte aligned rows in shared memory)
        const float4* lse4 = reinterpret_cast<const float4*>(smem + OFF_ROWV) + (s * 2 * BQ + 32 * half) / 4;
        float lse[32], dlt[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 a = lse4[k], d = lse4[k + BQ / 4];
          lse[4 * k + 0] = a.x;
          lse[4 * k + 1] = a.y;
          lse[4 * k + 2] = a.z;
          lse[4 * k + 3] = a.w;
          dlt[4 * k + 0] = d.x;
          dlt[4 * k + 1] = d.y;
          dlt[4 * k + 2] = d.z;
          dlt[4 * k + 3] = d.w;
        }
        const uint32_t s_addr = tmem + COL_S + 64u * (gs & 1) + lane_off;
        float pr[32];
        {
          uint32_t u[32];
          tmem_ld32(s_addr + 32 * half, u);
          tmem_wait_ld();
          if (qc >= q_min) {  // every query of the half-tile sees this key
#pragma unroll
            for (int k = 0; k < 32; ++k) pr[k] = ex2_approx(fmaf(__uint_as_float(u[k]), p.scale_log2, -lse[k]));
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              pr[k] = qc + k >= q_min ? ex2_approx(fmaf(__uint_as_float(u[k]), p.scale_log2, -lse[k])) : 0.f;
          }
        }
        {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(pr[2 * k], pr[2 * k + 1]);
          // P^T packed in place over this half's own score columns (query pair k -> column
          // 32*half + k), so the other warpgroup's scores are never overwritten unread
          tmem_st16(s_addr + 32 * half, w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[gs & 1]);
        if (lane == 0) LAGA_TRACE_POINT(dkdv, 11, gs);
        if (!warp_wait(dp_full, gs & 1, 63)) { ok = false; break; }
        if (lane == 0) LAGA_TRACE_POINT(dkdv, 12, gs);
        tc_fence_after();
        const uint32_t dp_addr = tmem + COL_DP + lane_off;
        {
          uint32_t u[32];
          tmem_ld32(dp_addr + 32 * half, u);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dp_free);  // dP(i+1) may overwrite the dP^T columns
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_bf16x2(pr[2 * k] * (__uint_as_float(u[2 * k]) - dlt[2 * k]),
                               pr[2 * k + 1] * (__uint_as_float(u[2 * k + 1]) - dlt[2 * k + 1]));
          // dS^T packed over this half's second 16 score columns of S^T(i) (already read)
          tmem_st16(s_addr + 32 * half + 16, w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full(gs));
        if (lane == 0) LAGA_TRACE_POINT(dkdv, 13, gs);
      }
      if (!ok || !warp_wait(dv_done, u & 1, 65)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t a[32], c[32];
        drain_load(false, a, c);
        tmem_wait_ld();
        drain_put(h, false, a, c);
      }
      if (!warp_wait(acc_done, u & 1, 64)) { ok = false; break; }
      if (lane == 0) LAGA_TRACE_POINT(dkdv, 29, u);
      tc_fence_after();
      {
        uint32_t a[32], c[32];
        drain_load(true, a, c);
        tmem_wait_ld();
        if (u + 1 < G) {
          // dK_nope restarts from zero for the next head (its first dK accumulates);
          // its values are in registers, so the accumulators can be released first
          uint32_t zero[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) zero[k] = 0u;
          tmem_st32(tmem + lane_off + COL_DK + 64 * half, zero);
          tmem_st32(tmem + lane_off + COL_DK + 64 * half + 32, zero);
          tmem_wait_st();
          release(acc_free);
        }
        drain_put(h, true, a, c);
      }
      if (lane == 0) LAGA_TRACE_POINT(dkdv, 27, u);
      if (u + 1 == G) {
        // the RoPE-key gradient summed over this group's heads: fp32 partial hg,
        // columns [32*half, 32*half + 32) as two 16-column (64-byte) chunks
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + COL_DK + 128 + 32 * half, v);
        tmem_wait_ld();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = z ? 0u : __float_as_uint(__uint_as_float(v[16 * hh + k]) * p.scale);
          put_chunk(w, &mdKR, hg * 64 + 32 * half + 16 * hh);
        }
      }
    }
    if (lane == 0) bulk_wait_read_all();  // shared memory must not go away under a store
  }

  LAGA_TRACE_POINT(dkdv, 28, 0);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) publish_abort(abort_flag, p.status);
  LAGA_TRACE_POINT(dkdv, 31, 0);
  LAGA_TRACE_CTA_END(dkdv);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

LaunchResult tc_attn_bwd_dkdv(const Dims& d, const bf16* q, const bf16* k_rope, const bf16* dout,
                              const BwdWorkspace& w, cudaStream_t st) {
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
  // the drain's stores: [32 rows][64 bytes] boxes, 64-byte swizzle, of dK_nope and dV
  // ([B * skv_pad rows][n_h * 128] bf16) and of the RoPE-key partials
  // ([B * skv_pad rows][n_h / G * 64] fp32)
  CUtensorMap mdK, mdV, mdKR;
  const int G = dkdv_heads_per_cta(d.n_h);
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t dims[2] = {kv_inner, kv_rows};
    const uint64_t strides[1] = {kv_inner * 2};
    const uint32_t box[2] = {32, 32};
    r.cu = make_tmap(&mdK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.dk_ws, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_64B);
    if (r.cu == CUDA_SUCCESS)
      r.cu = make_tmap(&mdV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.dv_ws, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_64B);
  }
  if (r.cu == CUDA_SUCCESS) {
    const uint64_t inner = static_cast<uint64_t>(d.n_h / G) * 64;
    const uint64_t dims[2] = {inner, kv_rows};
    const uint64_t strides[1] = {inner * 4};
    const uint32_t box[2] = {16, 32};
    r.cu = make_tmap(&mdKR, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, w.dkr_ws, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_64B);
  }
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps attention backward (dK, dV)";
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
  p.scale = d.scale;
  p.scale_log2 = d.scale * 1.4426950408889634f;
  p.lse2 = w.lse2;
  p.delta = w.delta;
  p.G = G;
  p.n_hg = d.n_h / G;
  p.successor = sm_count();
  r.err = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(attn_bwd_dkdv)";
    return r;
  }
  attn_bwd_dkdv_kernel<<<dim3(d.skv_pad / BKV, p.n_hg, d.B), NTHREADS, SMEM_BYTES, st>>>(mQ, mK, mR, mV, mdO, mdK, mdV, mdKR, p);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "attn_bwd_dkdv_kernel launch";
  return r;
}

}  // namespace laga
