// Tensor-core (tcgen05 + TMEM + TMA) GEMMs of the K/V reconstruction and its
// backward, for bf16 operands with fp32 accumulation:
//
//   K/V rebuild  K_nope = c_kv W_UK, V = c_kv W_UV           per batch element
//                (LAGA: per-head K/V rebuilt locally from the gathered latent)
//   DCKV         dc_kv = dK_nope W_UK^T + dV W_UV^T          per batch element
//   DW           dW_UK = sum_b c_kv[b]^T dK_nope[b], dW_UV likewise
//   QLAT         q_lat_h = q_nope_h W_UK_h^T       per head (the absorbed form's query)
//   OUTPROJ      out_h = ctx_h W_UV_h              per head (the absorbed form's output)
//
// The K/V rebuild has a kernel of its own (recon_tmem_a_kernel, below: the
// latent tile is a TMEM operand). One persistent kernel template serves the
// others. Warp roles (224 threads):
//   warp 0      TMA producer of the A tiles into a STAGES-deep shared-memory ring
//   warp 1      TMEM allocator; the whole warp runs the MMA issue loop
//   warps 2..5  epilogue: TMEM -> registers -> bf16 -> shared memory -> tensor-map
//               store, per warp in [32 rows][32 cols] boxes through two buffers
//   warp 6      TMA producer of the B tiles
// Two TMEM accumulators let the epilogue of one tile overlap the next tile's
// main loop. Operand tiles use the 128-byte swizzle; a K-major tile is
// [rows][64 K] (128-byte rows), an MN-major tile is a set of [64 K][64 MN] boxes.
#include "internal.h"
#include "ptx.cuh"

#include <algorithm>

LAGA_TRACE_DEFINE(gemm)

namespace laga {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
enum Mode { DCKV = 1, DW = 2, QLAT = 3, OUTPROJ = 4 };

struct GemmParams {
  int* status;  // device status word (timeouts)
  int m_tiles, n_tiles, batches;  // tiles = m_tiles * n_tiles * batches, n fastest
  int n_tiles_first;              // K/V rebuild / DW: n tiles served by operand pair 0
  int k_blocks;                   // BK-blocks per tile
  int kb_first;                   // DCKV: k blocks served by pair 0 (dK_nope . W_UK^T)
  int kb_per_batch;               // DW: k blocks per batch element
  int S, skv_pad;
  bf16* out0;
  bf16* out1;
  long long ldo;               // elements per output row
  long long out_batch_stride;  // elements between batch elements of the output
  int rows_valid;              // output rows (per batch element) that exist
  int d_lat;                   // QLAT: latent width (output columns per head)
  int a_head_stride;           // QLAT / OUTPROJ: A columns between heads
  int b_head_stride;           // QLAT: B columns between heads
  int m_first;                 // K/V rebuild: first 128-row tile (a row range of the latent)
};

// Tile order: within a batch element, bands of GROUP_M m-tiles are walked n by n
// (m fastest inside a band). The CTAs running at one time then cover a block of
// about GROUP_M x (SMs / GROUP_M) tiles, so each A and B tile is wanted by a few
// CTAs at once instead of an m-row of 128 CTAs all asking L2 for the same A tile.
constexpr int GROUP_M = 8;

__device__ __forceinline__ void tile_coords(const GemmParams& p, int tile, int& b, int& m, int& n) {
  const int tiles_per_batch = p.m_tiles * p.n_tiles;
  b = tile / tiles_per_batch;
  const int t = tile - b * tiles_per_batch;
  const int per_band = GROUP_M * p.n_tiles;
  const int band = t / per_band;
  const int first_m = band * GROUP_M;
  const int gm = min(p.m_tiles - first_m, GROUP_M);
  const int r = t - band * per_band;
  m = first_m + r % gm;
  n = r / gm;
}

// MH = 2 makes a tile 256 rows tall: two M = 128 products per K16 step share
// each B k-block, so a stage streams 64 KB per 1024 tensor cycles (64 B/clk)
// instead of 48 KB per 512 (94 B/clk). Its two accumulators fill TMEM, so the
// epilogue of a tile does not overlap the next one's main loop; that costs
// little where the k loop is long (DCKV, DW).
template <int MODE, int BN, int STAGES, int MH = 1>
struct Cfg {
  static constexpr int A_HALF = BM * BK * 2;
  static constexpr int A_BYTES = MH * A_HALF;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_BYTES = 256;
  // epilogue staging: 4 warps x 2 buffers x [32 rows][32 bf16] (64-byte swizzle)
  static constexpr int EPI_BYTES = 4 * 2 * 32 * 64;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + BAR_BYTES;
  static constexpr int NACC = (2 * MH * BN <= 512) ? 2 : 1;  // accumulator sets in TMEM
  static constexpr uint32_t TMEM_COLS = NACC * MH * BN;
  static constexpr bool A_MN = (MODE == DW);
  static constexpr bool B_MN = (MODE != DCKV && MODE != QLAT);
  static constexpr uint32_t IDESC = idesc_bf16(BM, BN, A_MN, B_MN);
  static_assert(TMEM_COLS <= 512, "the accumulators must fit in TMEM");
  static_assert(BN % 64 == 0 && BN <= 256, "BN");
  static_assert(MH == 1 || MODE == DCKV || MODE == DW, "256-row tiles serve the long-k GEMMs");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// One epilogue warp's share of a finished tile: TMEM lanes 32*quarter .. +31 of
// MH accumulators of BN columns (t_acc = the first one's column), i.e. rows
// y_tile + 128*h + 32*quarter .. +31 of the output, written as [32 rows][32 cols]
// bf16 boxes: a 32-column chunk goes TMEM -> registers -> bf16 -> one of the
// warp's two shared-memory buffers (64-byte swizzle) -> a tensor-map store issued
// by lane 0. After the last chunk has been read from TMEM the warp arrives on
// acc_empty. chunk counts the warp's chunks so far (buffer = chunk % NBUF).
constexpr int EPI_BOX = 32 * 64;

template <int BN, int MH, int NBUF = 2>
__device__ __forceinline__ void epilogue_tile(uint32_t t_acc, int quarter, int lane, const CUtensorMap* omap, int n0,
                                              int y_tile, int b, uint8_t* ebuf, int& chunk, uint64_t* acc_empty) {
#pragma unroll 1
  for (int h = 0; h < MH; ++h) {
    const int y0 = y_tile + h * BM + quarter * 32;  // first row of this warp's boxes
    const uint32_t t_row = t_acc + h * BN + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32, ++chunk) {
      uint32_t r[32];
      tmem_ld32(t_row + c0, r);
      tmem_wait_ld();
      if (h == MH - 1 && c0 + 32 == BN) {  // the accumulator has been read out: the MMA may reuse it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      }
      uint8_t* box = ebuf + (chunk % NBUF) * EPI_BOX;
      if (lane == 0) bulk_wait_read_n<NBUF - 1>();  // the store that last read this buffer is done reading
      __syncwarp();
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
        w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
        w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
        w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
        *reinterpret_cast<uint4*>(box + sw64_offset(lane, v)) = w;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(omap, box, n0 + c0, y0, b);
        bulk_commit_group();
      }
    }
  }
}

template <int MODE, int BN, int STAGES, int MH>
__global__ void __launch_bounds__(224, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapA1,
                   const __grid_constant__ CUtensorMap mapB0, const __grid_constant__ CUtensorMap mapB1,
                   const __grid_constant__ CUtensorMap mapO0, const __grid_constant__ CUtensorMap mapO1,
                   const GemmParams p) {
  using C = Cfg<MODE, BN, STAGES, MH>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  uint8_t* sEpi = smem + STAGES * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + C::EPI_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int tiles_per_batch = p.m_tiles * p.n_tiles;
  const int num_tiles = tiles_per_batch * p.batches;

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // Two producers, in different warps: warp 0 loads the A tiles, warp 6 the B
      // tiles, each announcing its own bytes on the stage's full barrier (count 2).
      // One thread issuing both streams tops out well below the fill rate the SM
      // can take; copies from separate threads proceed side by side.
      const bool load_a = warp == 0;
      if (load_a) {
        tma_prefetch_desc(&mapA0);
        tma_prefetch_desc(&mapA1);
      } else {
        tma_prefetch_desc(&mapB0);
        tma_prefetch_desc(&mapB1);
      }
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int b, m, n;
        tile_coords(p, tile, b, m, n);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait_or_abort(&empty[s], ph ^ 1, abort_flag, 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], load_a ? C::A_BYTES : C::B_BYTES);
          uint8_t* a = sA + s * C::A_BYTES;
          uint8_t* bsm = sB + s * C::B_BYTES;
          if constexpr (MODE == DCKV) {
            const bool second = kb >= p.kb_first;
            const int kk = second ? kb - p.kb_first : kb;
            if (load_a)  // one [BM*MH rows][64] box
              tma_load_2d(a, second ? &mapA1 : &mapA0, &full[s], kk * BK, b * p.skv_pad + m * BM * MH);
            else
              tma_load_2d(bsm, second ? &mapB1 : &mapB0, &full[s], kk * BK, n * BN);
          } else if constexpr (MODE == QLAT) {
            // tile n covers latent columns [n*BN, n*BN + BN) of head (n*BN) / d_c
            const int h = (n * BN) / p.d_lat;
            const int c0 = n * BN - h * p.d_lat;
            if (load_a)
              tma_load_2d(a, &mapA0, &full[s], h * p.a_head_stride + kb * BK, m * BM);
            else
              tma_load_2d(bsm, &mapB0, &full[s], h * p.b_head_stride + kb * BK, c0);
          } else if constexpr (MODE == OUTPROJ) {
            // tile n is head n (BN = the head's value width)
            if (load_a) {
              tma_load_2d(a, &mapA0, &full[s], n * p.a_head_stride + kb * BK, m * BM);
            } else {
#pragma unroll
              for (int i = 0; i < BN / 64; ++i)
                tma_load_2d(bsm + i * 8192, &mapB0, &full[s], n * BN + 64 * i, kb * BK);
            }
          } else {
            const bool second = n >= p.n_tiles_first;
            const int n0 = (second ? n - p.n_tiles_first : n) * BN;
            const int bb = kb / p.kb_per_batch;
            const int kk = kb - bb * p.kb_per_batch;
            if (load_a) {
#pragma unroll
              for (int i = 0; i < 2 * MH; ++i)
                tma_load_2d(a + i * 8192, &mapA0, &full[s], m * BM * MH + 64 * i, bb * p.S + kk * BK);
            } else {
              const CUtensorMap* mb = second ? &mapB1 : &mapB0;
#pragma unroll
              for (int i = 0; i < BN / 64; ++i)
                tma_load_2d(bsm + i * 8192, mb, &full[s], n0 + 64 * i, bb * p.skv_pad + kk * BK);
            }
          }
        }
      }
      if (!ok) {
        // Let copies already in flight land before shared memory goes away.
        const int first = it > STAGES ? it - STAGES : 0;
        for (int j = first; j < it; ++j) mbar_drain(&full[j % STAGES], (j / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop; an elected lane issues. The barrier of
    // the next k-block (and, in a tile's last k-block, the next accumulator) is
    // tested without blocking between the current k-block's two pairs of MMAs,
    // so the check after them costs no shared-memory round trip behind the MMA
    // queue.
    int it = 0;
    int local = 0;
    bool ok = true;
    bool issued = false;
    uint32_t tf = 0, ta = 0;
    const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), C::A_MN ? 8192 : 16, 1024);
    const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), C::B_MN ? 8192 : 16, 1024);
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
      const int buf = local % C::NACC;
      const uint32_t use = static_cast<uint32_t>(local / C::NACC);
      if (!warp_wait_token(&acc_empty[buf], (use & 1) ^ 1, ta, abort_flag, 2)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * MH * BN;
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const int s = it % STAGES;
        if (!warp_wait_token(&full[s], (it / STAGES) & 1, tf, abort_flag, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t a_stage = a_desc0 + ((s * C::A_BYTES) >> 4);
        const uint64_t b_stage = b_desc0 + ((s * C::B_BYTES) >> 4);
        // the k-block's four K16 steps as two pairs, the next barriers tested between them
        constexpr uint32_t DA = (C::A_MN ? 2048 : 32) >> 4, DB = (C::B_MN ? 2048 : 32) >> 4;
        static_assert(BK == 64, "four K16 steps per k-block");
        // with MH = 2 each pair runs on both 128-row halves (A and D offset, B shared)
        constexpr uint32_t DH = C::A_HALF >> 4;
#pragma unroll
        for (int h = 0; h < MH; ++h)
          mma2_ss_warp(d_tmem + h * BN, a_stage + h * DH, a_stage + h * DH + DA, b_stage, b_stage + DB, C::IDESC,
                       kb != 0 ? 1u : 0u);
        tf = mbar_test(&full[(it + 1) % STAGES], ((it + 1) / STAGES) & 1);
        if (kb == p.k_blocks - 1) {
          const int nl = local + 1;
          ta = mbar_test(&acc_empty[nl % C::NACC], ((static_cast<uint32_t>(nl / C::NACC)) & 1) ^ 1);
        }
#pragma unroll
        for (int h = 0; h < MH; ++h)
          mma2_ss_warp(d_tmem + h * BN, a_stage + h * DH + 2 * DA, a_stage + h * DH + 3 * DA, b_stage + 2 * DB,
                       b_stage + 3 * DB, C::IDESC, 1u);
        issued = true;
        mma_commit_warp(&empty[s]);
      }
      if (ok) mma_commit_warp(&acc_full[buf]);
    }
    if (!ok && issued) {
      mma_commit_warp(drain);
      if (lane == 0) mbar_drain(drain, 0);
      __syncwarp();
    }
  } else {
    // Epilogue warps 2..5: warp (w % 4) may read TMEM lanes 32*(w%4) .. +31.
    // Each warp writes its 32 rows of a tile as [32 rows][32 cols] boxes: a
    // 32-column chunk goes TMEM -> registers -> bf16 -> one of the warp's two
    // shared-memory buffers (64-byte swizzle) -> a tensor-map store issued by lane
    // 0. Measured on GB300: row-per-thread 16-byte global stores from all SMs at
    // once run at ~64 cycles per warp instruction, coalesced ones at ~24; the
    // K/V rebuild writes 1 GB, so its epilogue set the pace with direct stores.
    const int quarter = warp & 3;
    uint8_t* ebuf = sEpi + (warp - 2) * 2 * EPI_BOX;
    const CUtensorMap* map0 = &mapO0;
    const CUtensorMap* map1 = &mapO1;
    if (lane == 0) {
      tma_prefetch_desc(map0);
      tma_prefetch_desc(map1);
    }
    int local = 0;
    int chunk = 0;  // chunks stored by this warp so far (buffer = chunk & 1)
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const int buf = local % C::NACC;
      const uint32_t use = static_cast<uint32_t>(local / C::NACC);
      bool ok = true;
      if (lane == 0) ok = mbar_wait_or_abort(&acc_full[buf], use & 1, abort_flag, 4);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      int b, m, n;
      tile_coords(p, tile, b, m, n);
      const CUtensorMap* omap;
      int n0;
      if constexpr (MODE == DCKV || MODE == QLAT || MODE == OUTPROJ) {
        omap = map0;
        n0 = n * BN;
      } else {
        const bool second = n >= p.n_tiles_first;
        omap = second ? map1 : map0;
        n0 = (second ? n - p.n_tiles_first : n) * BN;
      }
      epilogue_tile<BN, MH>(tmem_base + buf * MH * BN, quarter, lane, omap, n0, m * MH * BM, b, ebuf, chunk,
                            &acc_empty[buf]);
    }
    if (lane == 0) bulk_wait_read_all();  // shared memory must not go away under a store
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) publish_abort(abort_flag, p.status);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---- K/V rebuild with the latent tile as a TMEM operand
//
// K_nope, V = c_kv W_UK, c_kv W_UV have k = d_c = 512, so a tile's main loop is
// short, and with both operands streamed a 128 x 256 tile needs ~94 B/clk per SM
// from L2 (the SMs together get ~52). Here each CTA walks one contiguous range of
// (batch, m, n) tiles, n fastest, and holds the [128 rows][512] latent tile of
// the current m in TMEM (256 columns, bf16 pairs) as the A operand of TS-MMAs:
// only W streams, 16 KB per 256 tensor cycles (64 B/clk), through a 10-deep ring
// (160 KB in flight). Two 128-column accumulators let a tile's epilogue overlap
// the next one's main loop. When m changes, warp 0 brings the new latent tile in
// as eight [128][64] boxes through two shared-memory buffers and the epilogue
// warps move each row into TMEM (each thread owns one TMEM lane = one row), after
// every MMA that read the old tile has completed.
constexpr int TL_BN = 128;
constexpr int TL_DC = 512;
constexpr int TL_STAGES = 10;
constexpr int TL_B_BYTES = BK * TL_BN * 2;       // [64 K][128 N] as two [64][64] boxes
constexpr int TL_A_BOX = BM * BK * 2;            // one [128 rows][64] latent box
constexpr int TL_A_COL = 0;                      // TMEM columns of the latent tile
constexpr int TL_ACC_COL = TL_DC / 2;            // two accumulators after it
constexpr int TL_EPI_BUFS = 2;                   // store buffers per epilogue warp
constexpr int TL_SMEM = TL_STAGES * TL_B_BYTES + 2 * TL_A_BOX + 4 * TL_EPI_BUFS * EPI_BOX + 1024 + 512;
static_assert(TL_ACC_COL + 2 * TL_BN == 512, "TMEM budget");
static_assert(TL_SMEM <= 232448, "shared memory per CTA");

__global__ void __launch_bounds__(224, 1)
    recon_tmem_a_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB0,
                        const __grid_constant__ CUtensorMap mapB1, const __grid_constant__ CUtensorMap mapO0,
                        const __grid_constant__ CUtensorMap mapO1, const GemmParams p) {
  constexpr int STAGES = TL_STAGES;
  constexpr int KB = TL_DC / BK;          // k-blocks per tile
  constexpr int A_BOXES = TL_DC / BK;     // latent boxes per m
  constexpr uint32_t IDESC = idesc_bf16(BM, TL_BN, false, true);
  static_assert(KB % 2 == 0, "k-block pairs");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sB = smem;
  uint8_t* sAst = sB + STAGES * TL_B_BYTES;
  uint8_t* sEpi = sAst + 2 * TL_A_BOX;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + 4 * TL_EPI_BUFS * EPI_BOX);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = bars + 2 * STAGES + 2;
  uint64_t* ast_full = bars + 2 * STAGES + 4;   // latent staging buffer loaded
  uint64_t* ast_empty = bars + 2 * STAGES + 6;  // latent staging buffer read (4 warps)
  uint64_t* a_full = bars + 2 * STAGES + 8;     // latent tile in TMEM (4 warps)
  uint64_t* drain = bars + 2 * STAGES + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
      mbar_init(&ast_full[i], 1);
      mbar_init(&ast_empty[i], 4);
    }
    mbar_init(a_full, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // this CTA's contiguous tile range; the latent tile of tile t is key = t / n_tiles
  const int num_tiles = p.m_tiles * p.n_tiles * p.batches;
  const int per = num_tiles / gridDim.x, rem = num_tiles % gridDim.x;
  const int t_begin = blockIdx.x * per + min(static_cast<int>(blockIdx.x), rem);
  const int t_end = t_begin + per + (static_cast<int>(blockIdx.x) < rem ? 1 : 0);

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mapA);
      int boxes = 0, cur = -1;
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        const int key = t / p.n_tiles;
        if (key == cur) continue;
        cur = key;
        const int b = key / p.m_tiles, m = key - b * p.m_tiles + p.m_first;
        for (int i = 0; i < A_BOXES; ++i, ++boxes) {
          const int buf = boxes & 1;
          if (!mbar_wait_or_abort(&ast_empty[buf], ((boxes >> 1) & 1) ^ 1, abort_flag, 6)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&ast_full[buf], TL_A_BOX);
          tma_load_3d(sAst + buf * TL_A_BOX, &mapA, &ast_full[buf], i * BK, m * BM, b);
        }
      }
      if (!ok) {  // let copies in flight land before shared memory goes away
        for (int j = boxes > 2 ? boxes - 2 : 0; j < boxes; ++j) mbar_drain(&ast_full[j & 1], (j >> 1) & 1);
      }
    }
  } else if (warp == 6) {
    if (lane == 0) {
      tma_prefetch_desc(&mapB0);
      tma_prefetch_desc(&mapB1);
      int it = 0;
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        const int n = t % p.n_tiles;
        const bool second = n >= p.n_tiles_first;
        const int n0 = (second ? n - p.n_tiles_first : n) * TL_BN;
        const CUtensorMap* mb = second ? &mapB1 : &mapB0;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_or_abort(&empty[s], ((it / STAGES) & 1) ^ 1, abort_flag, 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], TL_B_BYTES);
          uint8_t* bsm = sB + s * TL_B_BYTES;
          tma_load_2d(bsm, mb, &full[s], n0, kb * BK);
          tma_load_2d(bsm + TL_B_BYTES / 2, mb, &full[s], n0 + 64, kb * BK);
        }
      }
      if (!ok) {
        const int first = it > STAGES ? it - STAGES : 0;
        for (int j = first; j < it; ++j) mbar_drain(&full[j % STAGES], (j / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // Two k-blocks per turn: their eight MMAs (512 tensor cycles) are queued before
    // the barriers of the next two stages are tested, so the tests' round trip
    // behind the MMA queue overlaps queued work.
    int it = 0, local = 0, a_uses = 0, cur = -1;
    bool ok = true;
    bool issued = false;
    uint32_t tf = 0, tf2 = 0, ta = 0;
    // B: MN-major [64 K][64 N] boxes, 8 KB apart; a K16 step is 16 rows of 128 bytes.
    const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), BK * 128, 1024);
    for (int t = t_begin; t < t_end && ok; ++t, ++local) {
      const int key = t / p.n_tiles;
      if (key != cur) {
        if (!warp_wait_or_abort(a_full, a_uses & 1, abort_flag, 5)) {
          ok = false;
          break;
        }
        tc_fence_after();
        ++a_uses;
        cur = key;
      }
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!warp_wait_token(&acc_empty[buf], (use & 1) ^ 1, ta, abort_flag, 2)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + TL_ACC_COL + buf * TL_BN;
      for (int kb = 0; kb < KB; kb += 2, it += 2) {
        const int s0 = it % STAGES, s1 = (it + 1) % STAGES;
        if (!warp_wait_token(&full[s0], (it / STAGES) & 1, tf, abort_flag, 3) ||
            !warp_wait_token(&full[s1], ((it + 1) / STAGES) & 1, tf2, abort_flag, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // latent K16 step k sits in TMEM columns 8k .. 8k+7
        const uint32_t a = tmem_base + TL_A_COL + kb * (BK / 2);
        const uint64_t b0 = b_desc0 + ((s0 * TL_B_BYTES) >> 4);
        const uint64_t b1 = b_desc0 + ((s1 * TL_B_BYTES) >> 4);
        constexpr uint32_t DB = 2048 >> 4;
        mma4_ts_warp(d_tmem, a, a + 8, a + 16, a + 24, b0, b0 + DB, b0 + 2 * DB, b0 + 3 * DB, IDESC,
                     kb != 0 ? 1u : 0u);
        mma4_ts_warp(d_tmem, a + 32, a + 40, a + 48, a + 56, b1, b1 + DB, b1 + 2 * DB, b1 + 3 * DB, IDESC, 1u);
        tf = mbar_test(&full[(it + 2) % STAGES], ((it + 2) / STAGES) & 1);
        tf2 = mbar_test(&full[(it + 3) % STAGES], ((it + 3) / STAGES) & 1);
        if (kb == KB - 2) {
          const int nl = local + 1;
          ta = mbar_test(&acc_empty[nl & 1], ((static_cast<uint32_t>(nl >> 1)) & 1) ^ 1);
        }
        issued = true;
        mma_commit_warp(&empty[s0]);
        mma_commit_warp(&empty[s1]);
      }
      if (!ok) break;
      mma_commit_warp(&acc_full[buf]);
    }
    if (!ok && issued) {
      mma_commit_warp(drain);
      if (lane == 0) mbar_drain(drain, 0);
      __syncwarp();
    }
  } else {
    // epilogue warps 2..5: warp (w % 4) owns TMEM lanes (= tile rows) 32*(w%4) .. +31
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint8_t* ebuf = sEpi + (warp - 2) * TL_EPI_BUFS * EPI_BOX;
    if (lane == 0) {
      tma_prefetch_desc(&mapO0);
      tma_prefetch_desc(&mapO1);
    }
    int boxes = 0;
    // Move the next latent tile from the staging buffers into TMEM columns
    // [0, 256): box i (K 64i .. 64i+63) -> columns 32i .. 32i+31, two bf16 per column.
    auto load_latent = [&]() -> bool {
      for (int i = 0; i < A_BOXES; ++i, ++boxes) {
        const int buf = boxes & 1;
        if (!warp_wait_or_abort(&ast_full[buf], (boxes >> 1) & 1, abort_flag, 7)) return false;
        const uint8_t* src = sAst + buf * TL_A_BOX + row * 128;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 128-byte swizzle: chunk c of row r sits at chunk c ^ (r % 8)
          const uint4 v = *reinterpret_cast<const uint4*>(src + ((c ^ (row & 7)) << 4));
          w[4 * c + 0] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        tmem_st32(tmem_base + TL_A_COL + 32 * i + lane_off, w);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ast_empty[buf]);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full);
      return true;
    };
    bool ok = t_begin < t_end ? load_latent() : true;
    int local = 0;
    int chunk = 0;
    for (int t = t_begin; t < t_end && ok; ++t, ++local) {
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!warp_wait_or_abort(&acc_full[buf], use & 1, abort_flag, 4)) break;
      tc_fence_after();
      const int key = t / p.n_tiles;
      // every MMA through tile t is done, so the latent columns may be replaced now
      if (t + 1 < t_end && (t + 1) / p.n_tiles != key && !load_latent()) break;
      const int n = t - key * p.n_tiles;
      const int b = key / p.m_tiles, m = key - b * p.m_tiles + p.m_first;
      const bool second = n >= p.n_tiles_first;
      const int n0 = (second ? n - p.n_tiles_first : n) * TL_BN;
      epilogue_tile<TL_BN, 1, TL_EPI_BUFS>(tmem_base + TL_ACC_COL + buf * TL_BN, quarter, lane, second ? &mapO1 : &mapO0, n0,
                              m * BM, b, ebuf, chunk, &acc_empty[buf]);
    }
    if (lane == 0) bulk_wait_read_all();  // shared memory must not go away under a store
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) publish_abort(abort_flag, p.status);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int MODE, int BN, int STAGES, int MH = 1>
LaunchResult launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                         const CUtensorMap& b1, const CUtensorMap& o0, const CUtensorMap& o1, const GemmParams& p,
                         cudaStream_t st) {
  using C = Cfg<MODE, BN, STAGES, MH>;
  LaunchResult r;
  auto kern = gemm_tc_kernel<MODE, BN, STAGES, MH>;
  r.err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(gemm)";
    return r;
  }
  const int tiles = p.m_tiles * p.n_tiles * p.batches;
  if (tiles == 0) return r;
  const int grid = std::min(tiles, sm_count());
  GemmParams pp = p;
  pp.status = device_status_ptr();
  kern<<<grid, 224, C::SMEM, st>>>(a0, a1, b0, b1, o0, o1, pp);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "gemm_tc_kernel launch";
  return r;
}

CUresult tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                      uint32_t box_inner, uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {row_bytes};
  const uint32_t box[2] = {box_inner, box_outer};
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

// Output map of the epilogue's [32 rows][32 cols] bf16 boxes (64-byte swizzle)
// over a [batches][rows][cols] tensor; rows beyond `rows` are clipped.
CUresult tmap_out(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t batches,
                  uint64_t batch_stride_elems) {
  const uint64_t dims[3] = {cols, rows, batches};
  const uint64_t strides[2] = {cols * 2, batch_stride_elems * 2};
  const uint32_t box[3] = {32, 32, 1};
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace

// Tile shape of the long-k GEMMs (dc_kv, dW): 256 x 256 tiles (MH = 2) move the
// fewest operand bytes per MMA but give few tiles; on small problems they leave
// most SMs idle. Take the widest shape whose tile count still fills about three
// quarters of the SMs: 256 x 256, else 128 x 256, else 128 x 128.
struct LongKShape {
  int MH, BN;
};
LongKShape long_k_shape(long long tiles_256x256, bool mh2_ok) {
  const long long fill = (3LL * sm_count()) / 4;
  if (mh2_ok && tiles_256x256 >= fill) return {2, 256};
  if (2 * tiles_256x256 >= fill) return {1, 256};
  return {1, 128};
}

LaunchResult tc_recon_fwd(const Dims& d, const bf16* c_kv, const bf16* W_UK, const bf16* W_UV, bf16* k_ws,
                          bf16* v_ws, int rows_pad, cudaStream_t st, int m_first, int m_count) {
  LaunchResult r;
  if (d.d_c != TL_DC) {  // the tensor-core path is planned only for d_c = 512
    r.err = cudaErrorInvalidValue;
    r.what = "K/V rebuild: d_c must be 512";
    return r;
  }
  CUtensorMap a0, b0, b1, o0, o1;
  const uint64_t N = static_cast<uint64_t>(d.n_h) * 128;
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(d.d_c), static_cast<uint64_t>(d.S),
                              static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {static_cast<uint64_t>(d.d_c) * 2, static_cast<uint64_t>(d.S) * d.d_c * 2};
    const uint32_t box[3] = {64, 128, 1};
    r.cu = make_tmap(&a0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c_kv, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    if (r.cu != CUDA_SUCCESS) {
      r.what = "tensor map c_kv";
      return r;
    }
  }
  r.cu = tmap_bf16_2d(&b0, W_UK, N, d.d_c, N * 2, 64, 64);  // [64 K][64 N] boxes
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_bf16_2d(&b1, W_UV, N, d.d_c, N * 2, 64, 64);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor map W";
    return r;
  }
  r.cu = tmap_out(&o0, k_ws, N, static_cast<uint64_t>(rows_pad), static_cast<uint64_t>(d.B),
                  static_cast<uint64_t>(rows_pad) * N);
  if (r.cu == CUDA_SUCCESS)
    r.cu = tmap_out(&o1, v_ws, N, static_cast<uint64_t>(rows_pad), static_cast<uint64_t>(d.B),
                    static_cast<uint64_t>(rows_pad) * N);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor map K/V out";
    return r;
  }
  r.err = cudaFuncSetAttribute(recon_tmem_a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TL_SMEM);
  if (r.err != cudaSuccess) {
    r.what = "cudaFuncSetAttribute(recon_tmem_a)";
    return r;
  }
  GemmParams p{};
  p.m_first = m_first;
  p.m_tiles = m_count < 0 ? rows_pad / BM : m_count;
  p.n_tiles_first = static_cast<int>(N / TL_BN);  // K_nope tiles, then as many V tiles
  p.n_tiles = 2 * p.n_tiles_first;
  p.batches = d.B;
  const int tiles = p.m_tiles * p.n_tiles * p.batches;
  if (tiles == 0) return r;
  p.status = device_status_ptr();
  recon_tmem_a_kernel<<<std::min(tiles, sm_count()), 224, TL_SMEM, st>>>(a0, b0, b1, o0, o1, p);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "recon_tmem_a_kernel launch";
  return r;
}

LaunchResult tc_recon_bwd_dc(const Dims& d, const bf16* dk_ws, const bf16* dv_ws, const bf16* W_UK,
                             const bf16* W_UV, bf16* dc_kv, cudaStream_t st) {
  // 256 x 256 tiles (two 128-row halves) stream 64 KB per 1024 tensor cycles;
  // 128 x 256 ones 48 KB per 512 and 128 x 128 ones 32 KB per 256. The k loop is
  // n_h * 256 long, so the unoverlapped epilogue of a 256-row tile is cheap.
  // A last 256-row tile that runs past a batch element's padded rows reads the
  // next element's (or zero-filled) rows; the output map clips those rows.
  LongKShape shape{1, 128};
  if (d.d_c % 256 == 0)
    shape = long_k_shape(static_cast<long long>(d.B) * ((d.skv_pad + 255) / 256) * (d.d_c / 256), true);
  const int BN = shape.BN, MH = shape.MH;
  LaunchResult r;
  CUtensorMap a0, a1, b0, b1;
  const uint64_t N = static_cast<uint64_t>(d.n_h) * 128;  // reduction length of each pair
  const uint64_t rows = static_cast<uint64_t>(d.B) * d.skv_pad;
  r.cu = tmap_bf16_2d(&a0, dk_ws, N, rows, N * 2, 64, 128 * MH);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_bf16_2d(&a1, dv_ws, N, rows, N * 2, 64, 128 * MH);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_bf16_2d(&b0, W_UK, N, d.d_c, N * 2, 64, BN);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_bf16_2d(&b1, W_UV, N, d.d_c, N * 2, 64, BN);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps dc_kv";
    return r;
  }
  GemmParams p{};
  p.m_tiles = (d.skv_pad + BM * MH - 1) / (BM * MH);
  p.n_tiles = d.d_c / BN;
  p.n_tiles_first = p.n_tiles;
  p.batches = d.B;
  p.kb_first = static_cast<int>(N / BK);
  p.k_blocks = 2 * p.kb_first;
  p.S = d.S;
  p.skv_pad = d.skv_pad;
  p.out0 = dc_kv;
  p.out1 = dc_kv;
  p.ldo = d.d_c;
  p.out_batch_stride = static_cast<long long>(d.S) * d.d_c;
  p.rows_valid = d.S;
  CUtensorMap o0;
  // Rows at or past the padded visible prefix are clipped: a 256-row tile may
  // overhang it, and the caller zero-fills those rows of dc_kv.
  r.cu = tmap_out(&o0, dc_kv, static_cast<uint64_t>(d.d_c), static_cast<uint64_t>(std::min(d.S, d.skv_pad)),
                  static_cast<uint64_t>(d.B), static_cast<uint64_t>(d.S) * d.d_c);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor map dc_kv out";
    return r;
  }
  if (MH == 2) return launch_gemm<DCKV, 256, 3, 2>(a0, a1, b0, b1, o0, o0, p, st);
  if (BN == 256) return launch_gemm<DCKV, 256, 4>(a0, a1, b0, b1, o0, o0, p, st);
  return launch_gemm<DCKV, 128, 6>(a0, a1, b0, b1, o0, o0, p, st);
}

LaunchResult tc_recon_bwd_dw(const Dims& d, const bf16* c_kv, const bf16* dk_ws, const bf16* dv_ws, bf16* dW_UK,
                             bf16* dW_UV, cudaStream_t st) {
  // 256-row tiles (two halves sharing each B k-block) when d_c allows them: the
  // k loop is B * S long, so the unoverlapped epilogue of such a tile is cheap.
  LongKShape shape{1, 128};
  if (d.n_h % 2 == 0)
    shape = long_k_shape(static_cast<long long>(d.d_c / 256) * 2 * (d.n_h / 2), d.d_c % 256 == 0);
  const int BN = shape.BN, MH = shape.MH;
  LaunchResult r;
  CUtensorMap a0, b0, b1;
  const uint64_t N = static_cast<uint64_t>(d.n_h) * 128;
  r.cu = tmap_bf16_2d(&a0, c_kv, d.d_c, static_cast<uint64_t>(d.B) * d.S, static_cast<uint64_t>(d.d_c) * 2, 64,
                      64);
  const uint64_t rows = static_cast<uint64_t>(d.B) * d.skv_pad;
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_bf16_2d(&b0, dk_ws, N, rows, N * 2, 64, 64);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_bf16_2d(&b1, dv_ws, N, rows, N * 2, 64, 64);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps dW";
    return r;
  }
  GemmParams p{};
  p.m_tiles = d.d_c / (BM * MH);
  p.n_tiles_first = static_cast<int>(N / BN);
  p.n_tiles = 2 * p.n_tiles_first;
  p.batches = 1;
  p.kb_per_batch = d.skv_pad / BK;
  p.k_blocks = p.kb_per_batch * d.B;
  p.S = d.S;
  p.skv_pad = d.skv_pad;
  p.out0 = dW_UK;
  p.out1 = dW_UV;
  p.ldo = static_cast<long long>(N);
  p.out_batch_stride = 0;
  p.rows_valid = d.d_c;
  CUtensorMap o0, o1;
  r.cu = tmap_out(&o0, dW_UK, N, static_cast<uint64_t>(d.d_c), 1, static_cast<uint64_t>(d.d_c) * N);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_out(&o1, dW_UV, N, static_cast<uint64_t>(d.d_c), 1, static_cast<uint64_t>(d.d_c) * N);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor map dW out";
    return r;
  }
  if (MH == 2) return launch_gemm<DW, 256, 3, 2>(a0, a0, b0, b1, o0, o1, p, st);
  if (BN == 256) return launch_gemm<DW, 256, 4>(a0, a0, b0, b1, o0, o1, p, st);
  return launch_gemm<DW, 128, 6>(a0, a0, b0, b1, o0, o1, p, st);
}

// ---- the absorbed MLA form's two projections (the rejected variant, run for comparison)

LaunchResult tc_absorbed_qlat(const Dims& d, const bf16* q, const bf16* W_UK, bf16* q_lat, cudaStream_t st) {
  LaunchResult r;
  CUtensorMap a0, b0, o0;
  const uint64_t rows = static_cast<uint64_t>(d.B) * d.Sq;
  const uint64_t qcols = static_cast<uint64_t>(d.n_h) * (d.d_nope + d.d_rope);
  const uint64_t lcols = static_cast<uint64_t>(d.n_h) * d.d_c;
  r.cu = tmap_bf16_2d(&a0, q, qcols, rows, qcols * 2, 64, 128);
  if (r.cu == CUDA_SUCCESS)
    r.cu = tmap_bf16_2d(&b0, W_UK, static_cast<uint64_t>(d.n_h) * d.d_nope, d.d_c,
                        static_cast<uint64_t>(d.n_h) * d.d_nope * 2, 64, 256);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_out(&o0, q_lat, lcols, rows, 1, rows * lcols);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps q_lat";
    return r;
  }
  GemmParams p{};
  p.m_tiles = static_cast<int>((rows + BM - 1) / BM);
  p.n_tiles = static_cast<int>(lcols / 256);
  p.n_tiles_first = p.n_tiles;
  p.batches = 1;
  p.k_blocks = d.d_nope / BK;
  p.d_lat = d.d_c;
  p.a_head_stride = d.d_nope + d.d_rope;
  p.b_head_stride = d.d_nope;
  return launch_gemm<QLAT, 256, 4>(a0, a0, b0, b0, o0, o0, p, st);
}

LaunchResult tc_absorbed_outproj(const Dims& d, const bf16* ctx, const bf16* W_UV, bf16* out, cudaStream_t st) {
  LaunchResult r;
  CUtensorMap a0, b0, o0;
  const uint64_t rows = static_cast<uint64_t>(d.B) * d.Sq;
  const uint64_t ccols = static_cast<uint64_t>(d.n_h) * d.d_c;
  const uint64_t ocols = static_cast<uint64_t>(d.n_h) * d.d_v;
  r.cu = tmap_bf16_2d(&a0, ctx, ccols, rows, ccols * 2, 64, 128);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_bf16_2d(&b0, W_UV, ocols, d.d_c, ocols * 2, 64, 64);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_out(&o0, out, ocols, rows, 1, rows * ocols);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor maps absorbed output";
    return r;
  }
  GemmParams p{};
  p.m_tiles = static_cast<int>((rows + BM - 1) / BM);
  p.n_tiles = d.n_h;
  p.n_tiles_first = p.n_tiles;
  p.batches = 1;
  p.k_blocks = d.d_c / BK;
  p.a_head_stride = d.d_c;
  return launch_gemm<OUTPROJ, 128, 6>(a0, a0, b0, b0, o0, o0, p, st);
}

}  // namespace laga
