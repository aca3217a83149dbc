// Tensor-core (tcgen05 + TMEM + TMA) GEMMs of the K/V reconstruction and its
// backward, for bf16 operands with fp32 accumulation:
//
//   RECON_FWD  K_nope = c_kv W_UK, V = c_kv W_UV           per batch element
//              (LAGA: per-head K/V rebuilt locally from the gathered latent)
//   DCKV       dc_kv = dK_nope W_UK^T + dV W_UV^T          per batch element
//   DW         dW_UK = sum_b c_kv[b]^T dK_nope[b], dW_UV likewise
//   QLAT       q_lat_h = q_nope_h W_UK_h^T       per head (the absorbed form's query)
//   OUTPROJ    out_h = ctx_h W_UV_h              per head (the absorbed form's output)
//
// One persistent kernel template serves all three. Warp roles (224 threads):
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
enum Mode { RECON_FWD = 0, DCKV = 1, DW = 2, QLAT = 3, OUTPROJ = 4 };

struct GemmParams {
  int* status;  // device status word (timeouts)
  int m_tiles, n_tiles, batches;  // tiles = m_tiles * n_tiles * batches, n fastest
  int n_tiles_first;              // RECON_FWD / DW: n tiles served by operand pair 0
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
  static constexpr int EPI_BOX = 32 * 64;
  static constexpr int EPI_BYTES = 4 * 2 * EPI_BOX;
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
          if (MODE == RECON_FWD && load_a && it < 512) LAGA_TRACE_POINT(gemm, 20, it);
          mbar_arrive_expect_tx(&full[s], load_a ? C::A_BYTES : C::B_BYTES);
          uint8_t* a = sA + s * C::A_BYTES;
          uint8_t* bsm = sB + s * C::B_BYTES;
          if constexpr (MODE == RECON_FWD) {
            const bool second = n >= p.n_tiles_first;
            const int n0 = (second ? n - p.n_tiles_first : n) * BN;
            if (load_a) {
              tma_load_3d(a, &mapA0, &full[s], kb * BK, m * BM, b);
            } else {
              const CUtensorMap* mb = second ? &mapB1 : &mapB0;
#pragma unroll
              for (int i = 0; i < BN / 64; ++i) tma_load_2d(bsm + i * 8192, mb, &full[s], n0 + 64 * i, kb * BK);
            }
          } else if constexpr (MODE == DCKV) {
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
        if (MODE == RECON_FWD && lane == 0 && it < 512) LAGA_TRACE_POINT(gemm, 1, it);
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
    const int row_in_tile = quarter * 32 + lane;
    uint8_t* ebuf = sEpi + (warp - 2) * 2 * C::EPI_BOX;
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
#pragma unroll 1
      for (int h = 0; h < MH; ++h) {
        const int y0 = (m * MH + h) * BM + quarter * 32;  // first row of this warp's boxes
        const uint32_t t_row = tmem_base + (buf * MH + h) * BN + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32, ++chunk) {
          uint32_t r[32];
          tmem_ld32(t_row + c0, r);
          tmem_wait_ld();
          if (h == MH - 1 && c0 + 32 == BN) {  // the accumulator has been read out: the MMA may reuse it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
          }
          uint8_t* box = ebuf + (chunk & 1) * C::EPI_BOX;
          if (lane == 0) bulk_wait_read_1();  // the store that last read this buffer is done reading
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
      if (MODE == RECON_FWD && lane == 0 && local < 512) LAGA_TRACE_POINT(gemm, 10, local);
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

LaunchResult tc_recon_fwd(const Dims& d, const bf16* c_kv, const bf16* W_UK, const bf16* W_UV, bf16* k_ws,
                          bf16* v_ws, int rows_pad, cudaStream_t st) {
  // n_h * 128 columns per weight: 256-wide tiles when they divide it, else 128.
  const int BN = (d.n_h % 2 == 0) ? 256 : 128;
  LaunchResult r;
  CUtensorMap a0, b0, b1;
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
  r.cu = tmap_bf16_2d(&b0, W_UK, N, d.d_c, N * 2, 64, 64);
  if (r.cu == CUDA_SUCCESS) r.cu = tmap_bf16_2d(&b1, W_UV, N, d.d_c, N * 2, 64, 64);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor map W";
    return r;
  }
  GemmParams p{};
  p.m_tiles = rows_pad / BM;
  p.n_tiles_first = static_cast<int>(N / BN);
  p.n_tiles = 2 * p.n_tiles_first;
  p.batches = d.B;
  p.k_blocks = d.d_c / BK;
  p.S = d.S;
  p.skv_pad = rows_pad;
  p.out0 = k_ws;
  p.out1 = v_ws;
  p.ldo = static_cast<long long>(N);
  p.out_batch_stride = static_cast<long long>(rows_pad) * N;
  p.rows_valid = rows_pad;
  CUtensorMap o0, o1;
  r.cu = tmap_out(&o0, k_ws, N, static_cast<uint64_t>(rows_pad), static_cast<uint64_t>(d.B),
                  static_cast<uint64_t>(rows_pad) * N);
  if (r.cu == CUDA_SUCCESS)
    r.cu = tmap_out(&o1, v_ws, N, static_cast<uint64_t>(rows_pad), static_cast<uint64_t>(d.B),
                    static_cast<uint64_t>(rows_pad) * N);
  if (r.cu != CUDA_SUCCESS) {
    r.what = "tensor map K/V out";
    return r;
  }
  if (BN == 256) return launch_gemm<RECON_FWD, 256, 4>(a0, a0, b0, b1, o0, o1, p, st);
  return launch_gemm<RECON_FWD, 128, 6>(a0, a0, b0, b1, o0, o1, p, st);
}

LaunchResult tc_recon_bwd_dc(const Dims& d, const bf16* dk_ws, const bf16* dv_ws, const bf16* W_UK,
                             const bf16* W_UV, bf16* dc_kv, cudaStream_t st) {
  // 256 x 256 tiles (two 128-row halves) stream 64 KB per 1024 tensor cycles;
  // 128 x 256 ones 48 KB per 512 and 128 x 128 ones 32 KB per 256. The k loop is
  // n_h * 256 long, so the unoverlapped epilogue of a 256-row tile is cheap.
  // A last 256-row tile that runs past a batch element's padded rows reads the
  // next element's (or zero-filled) rows; the output map clips those rows.
  const int BN = d.d_c % 256 == 0 ? 256 : 128;
  const int MH = BN == 256 ? 2 : 1;
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
  if (BN == 256) return launch_gemm<DCKV, 256, 3, 2>(a0, a1, b0, b1, o0, o0, p, st);
  return launch_gemm<DCKV, 128, 6>(a0, a1, b0, b1, o0, o0, p, st);
}

LaunchResult tc_recon_bwd_dw(const Dims& d, const bf16* c_kv, const bf16* dk_ws, const bf16* dv_ws, bf16* dW_UK,
                             bf16* dW_UV, cudaStream_t st) {
  // 256-row tiles (two halves sharing each B k-block) when d_c allows them: the
  // k loop is B * S long, so the unoverlapped epilogue of such a tile is cheap.
  const int BN = (d.n_h % 2 == 0) ? 256 : 128;
  const int MH = (BN == 256 && d.d_c % 256 == 0) ? 2 : 1;
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
