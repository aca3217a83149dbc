// CUDA-core path of the LAGA MLA attention block: fp32 arithmetic, any head
// widths. It serves fp32 problems (and bf16 on request) where the tensor-core
// kernels have no instance. Straightforward kernels: a tiled SIMT GEMM for the
// reconstruction contractions and one CTA per query row (forward, dq) or per
// latent row (dK, dV) for attention.
#include "internal.h"

#include <cmath>

namespace laga {
namespace {

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const bf16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float v) { *p = v; }
__device__ __forceinline__ void st(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

using ll = long long;

// C[m,n] = sum_k A(m,k) B(k,n) [+ sum_k A2(m,k) B2(k,n)], with element strides.
template <typename TA, typename TB, typename TO>
__global__ void __launch_bounds__(256) simt_gemm(int M, int N, int K, const TA* A, ll sam, ll sak, const TB* B,
                                                 ll sbk, ll sbn, int K2, const TA* A2, ll sam2, ll sak2,
                                                 const TB* B2, ll sbk2, ll sbn2, TO* Cp, ll scm, ll scn) {
  __shared__ float As[16][65];
  __shared__ float Bs[16][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int pass = 0; pass < 2; ++pass) {
    const int KK = pass == 0 ? K : K2;
    const TA* Ap = pass == 0 ? A : A2;
    const TB* Bp = pass == 0 ? B : B2;
    const ll am = pass == 0 ? sam : sam2, ak = pass == 0 ? sak : sak2;
    const ll bk = pass == 0 ? sbk : sbk2, bn = pass == 0 ? sbn : sbn2;
    if (Ap == nullptr || KK == 0) continue;
    for (int k0 = 0; k0 < KK; k0 += 16) {
      for (int e = threadIdx.x; e < 16 * 64; e += 256) {
        const int kk = e / 64, mm = e % 64;
        const int gm = m0 + mm, gk = k0 + kk;
        As[kk][mm] = (gm < M && gk < KK) ? ld(Ap + gm * am + gk * ak) : 0.f;
        const int gn = n0 + mm;
        Bs[kk][mm] = (gn < N && gk < KK) ? ld(Bp + gk * bk + gn * bn) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gm = m0 + ty * 4 + i, gn = n0 + tx * 4 + j;
      if (gm < M && gn < N) st(Cp + gm * scm + gn * scn, acc[i][j]);
    }
}

template <typename TA, typename TB, typename TO>
cudaError_t gemm(cudaStream_t st, int M, int N, int K, const TA* A, ll sam, ll sak, const TB* B, ll sbk, ll sbn,
                 TO* Cp, ll scm, ll scn, int K2 = 0, const TA* A2 = nullptr, ll sam2 = 0, ll sak2 = 0,
                 const TB* B2 = nullptr, ll sbk2 = 0, ll sbn2 = 0) {
  if (M == 0 || N == 0) return cudaSuccess;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  simt_gemm<TA, TB, TO><<<grid, 256, 0, st>>>(M, N, K, A, sam, sak, B, sbk, sbn, K2, A2, sam2, sak2, B2, sbk2,
                                              sbn2, Cp, scm, scn);
  return cudaGetLastError();
}

__device__ float block_reduce(float v, bool is_max, float* red) {
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float r = red[0];
  for (int i = 1; i < nw; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

// Score of local query i (in smem sq) against latent row j of head h.
template <typename T>
__device__ float score(const float* sq, const float* kn, const T* k_rope, const Dims& d, int b, int h, int j) {
  const float* kr = kn + ((static_cast<ll>(b) * d.S + j) * d.n_h + h) * d.d_nope;
  float s = 0.f;
  for (int k = 0; k < d.d_nope; ++k) s = fmaf(sq[k], kr[k], s);
  const T* rp = k_rope + (static_cast<ll>(b) * d.S + j) * d.d_rope;
  for (int k = 0; k < d.d_rope; ++k) s = fmaf(sq[d.d_nope + k], ld(rp + k), s);
  return s * d.scale;
}

// One CTA per (local query i, head h, batch b).
template <typename T>
__global__ void __launch_bounds__(128) simt_attn_fwd(Dims d, const T* q, const float* kn, const float* v,
                                                     const T* k_rope, T* out, float* lse) {
  extern __shared__ float sm[];
  float* red = sm;
  float* sq = sm + 32;
  float* ss = sq + d.d_qk();
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n_vis = d.causal ? d.q_offset + i + 1 : d.S;
  const T* qp = q + ((static_cast<ll>(b) * d.Sq + i) * d.n_h + h) * d.d_qk();
  for (int k = threadIdx.x; k < d.d_qk(); k += blockDim.x) sq[k] = ld(qp + k);
  __syncthreads();
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < n_vis; j += blockDim.x) {
    const float s = score(sq, kn, k_rope, d, b, h, j);
    ss[j] = s;
    mx = fmaxf(mx, s);
  }
  mx = block_reduce(mx, true, red);
  float sum = 0.f;
  for (int j = threadIdx.x; j < n_vis; j += blockDim.x) {
    const float e = expf(ss[j] - mx);
    ss[j] = e;
    sum += e;
  }
  sum = block_reduce(sum, false, red);
  const float inv = 1.f / sum;
  T* op = out + ((static_cast<ll>(b) * d.Sq + i) * d.n_h + h) * d.d_v;
  for (int c = threadIdx.x; c < d.d_v; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < n_vis; ++j) acc = fmaf(ss[j], v[((static_cast<ll>(b) * d.S + j) * d.n_h + h) * d.d_v + c], acc);
    st(op + c, acc * inv);
  }
  if (threadIdx.x == 0) lse[(static_cast<ll>(b) * d.n_h + h) * d.Sq + i] = mx + logf(sum);
}

// D[b,h,i] = dout_i . out_i
template <typename T>
__global__ void simt_delta(Dims d, const T* out, const T* dout, float* delta) {
  const ll row = static_cast<ll>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const ll rows = static_cast<ll>(d.B) * d.Sq * d.n_h;
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int c = lane; c < d.d_v; c += 32) acc = fmaf(ld(out + row * d.d_v + c), ld(dout + row * d.d_v + c), acc);
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  const int h = static_cast<int>(row % d.n_h);
  const ll bi = row / d.n_h;
  const int i = static_cast<int>(bi % d.Sq);
  const int b = static_cast<int>(bi / d.Sq);
  if (lane == 0) delta[(static_cast<ll>(b) * d.n_h + h) * d.Sq + i] = acc;
}

// dq for one (query i, head h, batch b).
template <typename T>
__global__ void __launch_bounds__(128) simt_attn_dq(Dims d, const T* q, const float* kn, const float* v,
                                                    const T* k_rope, const T* dout, const float* lse,
                                                    const float* delta, T* dq) {
  extern __shared__ float sm[];
  float* sq = sm;
  float* sdo = sq + d.d_qk();
  float* sds = sdo + d.d_v;
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n_vis = d.causal ? d.q_offset + i + 1 : d.S;
  const ll qrow = (static_cast<ll>(b) * d.Sq + i) * d.n_h + h;
  for (int k = threadIdx.x; k < d.d_qk(); k += blockDim.x) sq[k] = ld(q + qrow * d.d_qk() + k);
  for (int k = threadIdx.x; k < d.d_v; k += blockDim.x) sdo[k] = ld(dout + qrow * d.d_v + k);
  __syncthreads();
  const float L = lse[(static_cast<ll>(b) * d.n_h + h) * d.Sq + i];
  const float D = delta[(static_cast<ll>(b) * d.n_h + h) * d.Sq + i];
  for (int j = threadIdx.x; j < n_vis; j += blockDim.x) {
    const float p = expf(score(sq, kn, k_rope, d, b, h, j) - L);
    const float* vr = v + ((static_cast<ll>(b) * d.S + j) * d.n_h + h) * d.d_v;
    float dp = 0.f;
    for (int c = 0; c < d.d_v; ++c) dp = fmaf(sdo[c], vr[c], dp);
    sds[j] = p * (dp - D);
  }
  __syncthreads();
  for (int k = threadIdx.x; k < d.d_qk(); k += blockDim.x) {
    float acc = 0.f;
    if (k < d.d_nope) {
      for (int j = 0; j < n_vis; ++j) acc = fmaf(sds[j], kn[((static_cast<ll>(b) * d.S + j) * d.n_h + h) * d.d_nope + k], acc);
    } else {
      for (int j = 0; j < n_vis; ++j)
        acc = fmaf(sds[j], ld(k_rope + (static_cast<ll>(b) * d.S + j) * d.d_rope + (k - d.d_nope)), acc);
    }
    st(dq + qrow * d.d_qk() + k, acc * d.scale);
  }
}

// dK (no-RoPE part and this head's RoPE part) and dV for one (latent row j, head h, batch b).
template <typename T>
__global__ void __launch_bounds__(128) simt_attn_dkv(Dims d, const T* q, const float* kn, const float* v,
                                                     const T* k_rope, const T* dout, const float* lse,
                                                     const float* delta, float* dkn, float* dkr, float* dv) {
  extern __shared__ float sm[];
  float* sk = sm;
  float* svv = sk + d.d_qk();
  float* sp = svv + d.d_v;
  float* sds = sp + d.Sq;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const ll krow = (static_cast<ll>(b) * d.S + j) * d.n_h + h;
  for (int k = threadIdx.x; k < d.d_nope; k += blockDim.x) sk[k] = kn[krow * d.d_nope + k];
  for (int k = threadIdx.x; k < d.d_rope; k += blockDim.x)
    sk[d.d_nope + k] = ld(k_rope + (static_cast<ll>(b) * d.S + j) * d.d_rope + k);
  for (int k = threadIdx.x; k < d.d_v; k += blockDim.x) svv[k] = v[krow * d.d_v + k];
  __syncthreads();
  const int i0 = d.causal ? max(0, j - d.q_offset) : 0;
  for (int i = threadIdx.x; i < d.Sq; i += blockDim.x) {
    float p = 0.f, ds = 0.f;
    if (i >= i0) {
      const ll qrow = (static_cast<ll>(b) * d.Sq + i) * d.n_h + h;
      float s = 0.f;
      for (int k = 0; k < d.d_qk(); ++k) s = fmaf(ld(q + qrow * d.d_qk() + k), sk[k], s);
      p = expf(s * d.scale - lse[(static_cast<ll>(b) * d.n_h + h) * d.Sq + i]);
      float dp = 0.f;
      for (int c = 0; c < d.d_v; ++c) dp = fmaf(ld(dout + qrow * d.d_v + c), svv[c], dp);
      ds = p * (dp - delta[(static_cast<ll>(b) * d.n_h + h) * d.Sq + i]);
    }
    sp[i] = p;
    sds[i] = ds;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < d.d_v; c += blockDim.x) {
    float acc = 0.f;
    for (int i = i0; i < d.Sq; ++i) acc = fmaf(sp[i], ld(dout + ((static_cast<ll>(b) * d.Sq + i) * d.n_h + h) * d.d_v + c), acc);
    dv[krow * d.d_v + c] = acc;
  }
  for (int k = threadIdx.x; k < d.d_qk(); k += blockDim.x) {
    float acc = 0.f;
    for (int i = i0; i < d.Sq; ++i) acc = fmaf(sds[i], ld(q + ((static_cast<ll>(b) * d.Sq + i) * d.n_h + h) * d.d_qk() + k), acc);
    acc *= d.scale;
    if (k < d.d_nope)
      dkn[krow * d.d_nope + k] = acc;
    else
      dkr[krow * d.d_rope + (k - d.d_nope)] = acc;
  }
}

// dk_rope[b,j,:] = sum over heads of the per-head RoPE-key gradients.
template <typename T>
__global__ void simt_sum_heads(Dims d, const float* dkr, T* dk_rope) {
  const ll idx = static_cast<ll>(blockIdx.x) * blockDim.x + threadIdx.x;
  const ll total = static_cast<ll>(d.B) * d.S * d.d_rope;
  if (idx >= total) return;
  const int k = static_cast<int>(idx % d.d_rope);
  const ll bj = idx / d.d_rope;
  float acc = 0.f;
  for (int h = 0; h < d.n_h; ++h) acc += dkr[(bj * d.n_h + h) * d.d_rope + k];
  st(dk_rope + idx, acc);
}

struct SimtWs {
  float *kn, *v, *dkn, *dv, *dkr, *delta;
};

SimtWs carve(const Dims& d, void* ws, bool bwd) {
  SimtWs w{};
  char* p = static_cast<char*>(ws);
  auto take = [&](size_t n) {
    float* r = reinterpret_cast<float*>(p);
    p += align_up(n * sizeof(float), 256);
    return r;
  };
  const size_t rows = static_cast<size_t>(d.B) * d.S * d.n_h;
  w.kn = take(rows * d.d_nope);
  w.v = take(rows * d.d_v);
  if (bwd) {
    w.dkn = take(rows * d.d_nope);
    w.dv = take(rows * d.d_v);
    w.dkr = take(rows * d.d_rope);
    w.delta = take(static_cast<size_t>(d.B) * d.n_h * d.Sq);
  }
  return w;
}

size_t ws_bytes(const Dims& d, bool bwd) {
  const size_t rows = static_cast<size_t>(d.B) * d.S * d.n_h;
  size_t n = align_up(rows * d.d_nope * 4, 256) + align_up(rows * d.d_v * 4, 256);
  if (bwd)
    n += align_up(rows * d.d_nope * 4, 256) + align_up(rows * d.d_v * 4, 256) + align_up(rows * d.d_rope * 4, 256) +
         align_up(static_cast<size_t>(d.B) * d.n_h * d.Sq * 4, 256);
  return n;
}

template <typename T>
cudaError_t recon(const Dims& d, const T* c_kv, const T* W_UK, const T* W_UV, float* kn, float* v, cudaStream_t st) {
  const int M = d.B * d.S;
  const ll nk = static_cast<ll>(d.n_h) * d.d_nope, nv = static_cast<ll>(d.n_h) * d.d_v;
  cudaError_t e = gemm<T, T, float>(st, M, static_cast<int>(nk), d.d_c, c_kv, d.d_c, 1, W_UK, nk, 1, kn, nk, 1);
  if (e == cudaSuccess)
    e = gemm<T, T, float>(st, M, static_cast<int>(nv), d.d_c, c_kv, d.d_c, 1, W_UV, nv, 1, v, nv, 1);
  return e;
}

template <typename T>
LaunchResult fwd_t(const Dims& d, const T* q, const T* c_kv, const T* k_rope, const T* W_UK, const T* W_UV, T* out,
                   float* lse, void* ws, cudaStream_t st) {
  LaunchResult r;
  SimtWs w = carve(d, ws, false);
  r.err = recon(d, c_kv, W_UK, W_UV, w.kn, w.v, st);
  if (r.err != cudaSuccess) {
    r.what = "simt reconstruct";
    return r;
  }
  const size_t smem = (32 + d.d_qk() + d.S) * sizeof(float);
  auto k = simt_attn_fwd<T>;
  r.err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (r.err == cudaSuccess) {
    k<<<dim3(d.Sq, d.n_h, d.B), 128, smem, st>>>(d, q, w.kn, w.v, k_rope, out, lse);
    r.err = cudaGetLastError();
  }
  if (r.err != cudaSuccess) r.what = "simt attention forward";
  return r;
}

template <typename T>
LaunchResult bwd_t(const Dims& d, const T* q, const T* c_kv, const T* k_rope, const T* W_UK, const T* W_UV,
                   const T* out, const float* lse, const T* dout, T* dq, T* dc_kv, T* dk_rope, T* dW_UK, T* dW_UV,
                   void* ws, bool reuse_kv, cudaStream_t st) {
  LaunchResult r;
  SimtWs w = carve(d, ws, true);
  if (!reuse_kv) r.err = recon(d, c_kv, W_UK, W_UV, w.kn, w.v, st);
  if (r.err != cudaSuccess) {
    r.what = "simt reconstruct";
    return r;
  }
  const ll rows = static_cast<ll>(d.B) * d.Sq * d.n_h;
  simt_delta<T><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(d, out, dout, w.delta);
  const size_t smem_q = (d.d_qk() + d.d_v + d.S) * sizeof(float);
  const size_t smem_k = (d.d_qk() + d.d_v + 2 * d.Sq) * sizeof(float);
  auto kq = simt_attn_dq<T>;
  auto kk = simt_attn_dkv<T>;
  r.err = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_q));
  if (r.err == cudaSuccess)
    r.err = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_k));
  if (r.err != cudaSuccess) {
    r.what = "simt smem attribute";
    return r;
  }
  kq<<<dim3(d.Sq, d.n_h, d.B), 128, smem_q, st>>>(d, q, w.kn, w.v, k_rope, dout, lse, w.delta, dq);
  kk<<<dim3(d.S, d.n_h, d.B), 128, smem_k, st>>>(d, q, w.kn, w.v, k_rope, dout, lse, w.delta, w.dkn, w.dkr, w.dv);
  const ll nr = static_cast<ll>(d.B) * d.S * d.d_rope;
  if (nr > 0)  // no RoPE part (d_rope = 0): no RoPE-key gradient to sum
    simt_sum_heads<T><<<static_cast<unsigned>((nr + 255) / 256), 256, 0, st>>>(d, w.dkr, dk_rope);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) {
    r.what = "simt attention backward";
    return r;
  }
  const int M = d.B * d.S;
  const ll nk = static_cast<ll>(d.n_h) * d.d_nope, nv = static_cast<ll>(d.n_h) * d.d_v;
  // dc_kv = dK_nope W_UK^T + dV W_UV^T
  r.err = gemm<float, T, T>(st, M, d.d_c, static_cast<int>(nk), w.dkn, nk, 1, W_UK, 1, nk, dc_kv, d.d_c, 1,
                            static_cast<int>(nv), w.dv, nv, 1, W_UV, 1, nv);
  // dW = c_kv^T dK (sum over the batch folds into the reduction over B*S rows)
  if (r.err == cudaSuccess)
    r.err = gemm<T, float, T>(st, d.d_c, static_cast<int>(nk), M, c_kv, 1, d.d_c, w.dkn, nk, 1, dW_UK, nk, 1);
  if (r.err == cudaSuccess)
    r.err = gemm<T, float, T>(st, d.d_c, static_cast<int>(nv), M, c_kv, 1, d.d_c, w.dv, nv, 1, dW_UV, nv, 1);
  if (r.err != cudaSuccess) r.what = "simt reconstruction backward";
  return r;
}

}  // namespace

size_t simt_fwd_workspace(const Dims& d) { return ws_bytes(d, false); }
size_t simt_bwd_workspace(const Dims& d) { return ws_bytes(d, true); }

LaunchResult simt_reconstruct(const Dims& d, bool is_bf16, const void* c_kv, const void* W_UK, const void* W_UV,
                              void* k_nope, void* v, bool out_f32, cudaStream_t st) {
  LaunchResult r;
  const int M = d.B * d.S;
  const ll nk = static_cast<ll>(d.n_h) * d.d_nope, nv = static_cast<ll>(d.n_h) * d.d_v;
  if (is_bf16) {
    auto c = static_cast<const bf16*>(c_kv);
    if (out_f32) {
      r.err = gemm<bf16, bf16, float>(st, M, static_cast<int>(nk), d.d_c, c, d.d_c, 1, static_cast<const bf16*>(W_UK),
                                      nk, 1, static_cast<float*>(k_nope), nk, 1);
      if (r.err == cudaSuccess)
        r.err = gemm<bf16, bf16, float>(st, M, static_cast<int>(nv), d.d_c, c, d.d_c, 1,
                                        static_cast<const bf16*>(W_UV), nv, 1, static_cast<float*>(v), nv, 1);
    } else {
      r.err = gemm<bf16, bf16, bf16>(st, M, static_cast<int>(nk), d.d_c, c, d.d_c, 1, static_cast<const bf16*>(W_UK),
                                     nk, 1, static_cast<bf16*>(k_nope), nk, 1);
      if (r.err == cudaSuccess)
        r.err = gemm<bf16, bf16, bf16>(st, M, static_cast<int>(nv), d.d_c, c, d.d_c, 1,
                                       static_cast<const bf16*>(W_UV), nv, 1, static_cast<bf16*>(v), nv, 1);
    }
  } else {
    r.err = recon(d, static_cast<const float*>(c_kv), static_cast<const float*>(W_UK),
                  static_cast<const float*>(W_UV), static_cast<float*>(k_nope), static_cast<float*>(v), st);
  }
  if (r.err != cudaSuccess) r.what = "simt reconstruct";
  return r;
}

LaunchResult simt_fwd(const Dims& d, bool is_bf16, const void* q, const void* c_kv, const void* k_rope,
                      const void* W_UK, const void* W_UV, void* out, float* lse, void* ws, cudaStream_t st) {
  if (is_bf16)
    return fwd_t(d, static_cast<const bf16*>(q), static_cast<const bf16*>(c_kv), static_cast<const bf16*>(k_rope),
                 static_cast<const bf16*>(W_UK), static_cast<const bf16*>(W_UV), static_cast<bf16*>(out), lse, ws, st);
  return fwd_t(d, static_cast<const float*>(q), static_cast<const float*>(c_kv), static_cast<const float*>(k_rope),
               static_cast<const float*>(W_UK), static_cast<const float*>(W_UV), static_cast<float*>(out), lse, ws,
               st);
}

LaunchResult simt_bwd(const Dims& d, bool is_bf16, const void* q, const void* c_kv, const void* k_rope,
                      const void* W_UK, const void* W_UV, const void* out, const float* lse, const void* dout,
                      void* dq, void* dc_kv, void* dk_rope, void* dW_UK, void* dW_UV, void* ws, bool reuse_kv,
                      cudaStream_t st) {
  if (is_bf16)
    return bwd_t(d, static_cast<const bf16*>(q), static_cast<const bf16*>(c_kv), static_cast<const bf16*>(k_rope),
                 static_cast<const bf16*>(W_UK), static_cast<const bf16*>(W_UV), static_cast<const bf16*>(out), lse,
                 static_cast<const bf16*>(dout), static_cast<bf16*>(dq), static_cast<bf16*>(dc_kv),
                 static_cast<bf16*>(dk_rope), static_cast<bf16*>(dW_UK), static_cast<bf16*>(dW_UV), ws, reuse_kv,
                 st);
  return bwd_t(d, static_cast<const float*>(q), static_cast<const float*>(c_kv), static_cast<const float*>(k_rope),
               static_cast<const float*>(W_UK), static_cast<const float*>(W_UV), static_cast<const float*>(out), lse,
               static_cast<const float*>(dout), static_cast<float*>(dq), static_cast<float*>(dc_kv),
               static_cast<float*>(dk_rope), static_cast<float*>(dW_UK), static_cast<float*>(dW_UV), ws, reuse_kv,
               st);
}

}  // namespace laga
