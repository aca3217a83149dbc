// Internal launcher interfaces shared by the .cu files of the library.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace laga {

using bf16 = __nv_bfloat16;

// Problem sizes after validation (all counts fit in int32 on the device side).
struct Dims {
  int B, Sq, S, n_h, d_c, d_nope, d_rope, d_v, q_offset;
  // second query segment: rows i >= q_split (0: none) sit at q_offset2 + i - q_split
  int q_split, q_offset2;
  bool causal;
  float scale;  // softmax scale (natural-log domain)
  int skv_eff;  // latent rows the shard can see
  int skv_pad;  // skv_eff rounded up to the 128-row key tile
  int sq_pad;   // Sq rounded up to 128 (the forward and dq query tile; two 64-row dK/dV query tiles)
  __host__ __device__ int d_qk() const { return d_nope + d_rope; }
};

// Result of a launcher: cudaSuccess or the first error seen; `what` names the step.
struct LaunchResult {
  cudaError_t err = cudaSuccess;
  CUresult cu = CUDA_SUCCESS;
  const char* what = nullptr;
  bool ok() const { return err == cudaSuccess && cu == CUDA_SUCCESS; }
};

// Device address of this device's status word (timeouts of bounded waits);
// nullptr if it cannot be resolved.
int* device_status_ptr();
// Handle of the calling thread's current CUDA context (nullptr if none): the key,
// beside the device number, of the per-device caches of module symbol addresses.
void* current_context();
// Number of SMs of the current device (cached per device).
int sm_count();

// Sets the message laga_mla_last_error returns on this host thread.
void set_last_error(const char* msg);

// ---- tensor-map helper (driver entry point resolved once through the runtime)
CUresult make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                   const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                   CUtensorMapSwizzle swizzle);

// ---- SIMT (CUDA-core, fp32 math) path: any dims.
size_t simt_fwd_workspace(const Dims& d);
size_t simt_bwd_workspace(const Dims& d);
LaunchResult simt_reconstruct(const Dims& d, bool is_bf16, const void* c_kv, const void* W_UK, const void* W_UV,
                              void* k_nope, void* v, bool out_f32, cudaStream_t st);
LaunchResult simt_fwd(const Dims& d, bool is_bf16, const void* q, const void* c_kv, const void* k_rope,
                      const void* W_UK, const void* W_UV, void* out, float* lse, void* ws, cudaStream_t st);
LaunchResult simt_bwd(const Dims& d, bool is_bf16, const void* q, const void* c_kv, const void* k_rope,
                      const void* W_UK, const void* W_UV, const void* out, const float* lse, const void* dout,
                      void* dq, void* dc_kv, void* dk_rope, void* dW_UK, void* dW_UV, void* ws, bool reuse_kv,
                      cudaStream_t st);

// ---- tensor-core path (bf16, d_c=512, d_nope=d_v=128, d_rope=64).
bool tc_supported(const Dims& d);
size_t tc_fwd_workspace(const Dims& d);
size_t tc_bwd_workspace(const Dims& d);

// K_nope/V for rows [0, rows) of every batch element into [B][rows_pad][n_h*128] bf16
// (rows_pad a multiple of 128; rows beyond S come out zero).
// K_nope / V of latent row tiles [m_first, m_first + m_count) (128 rows each; all of
// [0, rows_pad / 128) when m_count < 0) into the [B][rows_pad][n_h * 128] buffers.
LaunchResult tc_recon_fwd(const Dims& d, const bf16* c_kv, const bf16* W_UK, const bf16* W_UV, bf16* k_ws,
                          bf16* v_ws, int rows_pad, cudaStream_t st, int m_first = 0, int m_count = -1);
// dc_kv = dK_nope W_UK^T + dV W_UV^T (rows < S; rows >= skv_pad zeroed)
LaunchResult tc_recon_bwd_dc(const Dims& d, const bf16* dk_ws, const bf16* dv_ws, const bf16* W_UK,
                             const bf16* W_UV, bf16* dc_kv, cudaStream_t st);
// dW_UK = sum_b c_kv[b]^T dK_nope[b], dW_UV likewise.
LaunchResult tc_recon_bwd_dw(const Dims& d, const bf16* c_kv, const bf16* dk_ws, const bf16* dv_ws, bf16* dW_UK,
                             bf16* dW_UV, cudaStream_t st);

LaunchResult tc_attn_fwd(const Dims& d, const bf16* q, const bf16* k_ws, const bf16* v_ws, const bf16* k_rope,
                         bf16* out, float* lse, cudaStream_t st);
LaunchResult tc_attn_fwd_fused(const Dims& d, const bf16* q, const bf16* c_kv, const bf16* W_UK,
                               const bf16* W_UV, const bf16* k_rope, bf16* out, float* lse, cudaStream_t st);

struct BwdWorkspace {
  bf16* k_ws;       // [B][skv_pad][n_h*128]
  bf16* v_ws;       // [B][skv_pad][n_h*128]
  bf16* dk_ws;      // [B][skv_pad][n_h*128]
  bf16* dv_ws;      // [B][skv_pad][n_h*128]
  float* dkr_ws;    // [B][skv_pad][n_h / G][64]  RoPE-key gradient per head group (fp32)
  float* lse2;      // [B][n_h][sq_pad]  lse * log2(e), +inf on padded rows
  float* delta;     // [B][n_h][sq_pad]  rowsum(dout * out), 0 on padded rows
};
BwdWorkspace tc_bwd_carve(const Dims& d, void* ws);
// Heads per dK/dV CTA (G): the CTA walks G consecutive heads of one key tile and
// sums their RoPE-key gradients in TMEM, so the workspace holds n_h / G partials.
int dkdv_heads_per_cta(int n_h);

LaunchResult tc_bwd_pre(const Dims& d, const bf16* out, const bf16* dout, const float* lse, const BwdWorkspace& w,
                        cudaStream_t st);
// dV, dK_nope (bf16) and per-head RoPE-key gradients (fp32) into the workspace.
LaunchResult tc_attn_bwd_dkdv(const Dims& d, const bf16* q, const bf16* k_rope, const bf16* dout,
                              const BwdWorkspace& w, cudaStream_t st);
// dq, written once per element from a TMEM accumulator.
LaunchResult tc_attn_bwd_dq(const Dims& d, const bf16* q, const bf16* k_rope, const bf16* dout,
                            const BwdWorkspace& w, bf16* dq, cudaStream_t st);
// dk_rope = sum over heads of the per-head RoPE-key gradients.
LaunchResult tc_bwd_post(const Dims& d, const BwdWorkspace& w, bf16* dk_rope, cudaStream_t st);

// ---- the absorbed MLA form (for comparison; bf16, the tensor-core dims).
// q_lat [B*Sq][n_h*d_c] = per head q_nope_h W_UK_h^T
LaunchResult tc_absorbed_qlat(const Dims& d, const bf16* q, const bf16* W_UK, bf16* q_lat, cudaStream_t st);
// ctx [B*Sq][n_h*d_c] (attention in latent space) and lse, from q_lat, q's RoPE part, c_kv, k_rope
LaunchResult tc_absorbed_attn(const Dims& d, const bf16* q_lat, const bf16* q, const bf16* c_kv, const bf16* k_rope,
                              bf16* ctx, float* lse, cudaStream_t st);
// out [B*Sq][n_h*d_v] = per head ctx_h W_UV_h
LaunchResult tc_absorbed_outproj(const Dims& d, const bf16* ctx, const bf16* W_UV, bf16* out, cudaStream_t st);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace laga
