// Workspace layout and the small memory-bound kernels around the tensor-core
// attention backward:
//   pre   D_i = dout_i . out_i and lse in the log2 domain, padded per (b, h) row
//   post  dk_rope = sum of the RoPE-key gradient partials, one per head group of
//         the dK/dV kernel (the RoPE key is one tensor shared by every head, so its
//         gradient collects all of them)
#include "internal.h"

namespace laga {

// The fixed head dims of the tensor-core kernels; their tensor-map row coordinates
// (batch * padded rows) are 32-bit.
bool tc_supported(const Dims& d) {
  const int64_t rows_lim = int64_t(1) << 31;
  return d.d_c == 512 && d.d_nope == 128 && d.d_v == 128 && d.d_rope == 64 &&
         static_cast<int64_t>(d.B) * d.skv_pad < rows_lim && static_cast<int64_t>(d.B) * d.sq_pad < rows_lim &&
         static_cast<int64_t>(d.B) * d.S < rows_lim;
}

int dkdv_heads_per_cta(int n_h) { return n_h % 4 == 0 ? 4 : (n_h % 2 == 0 ? 2 : 1); }

namespace {
size_t kv_ws_bytes(const Dims& d) { return align_up(static_cast<size_t>(d.B) * d.skv_pad * d.n_h * 128 * 2, 256); }
}  // namespace

size_t tc_fwd_workspace(const Dims& d) { return 2 * kv_ws_bytes(d); }

size_t tc_bwd_workspace(const Dims& d) {
  const size_t kv = kv_ws_bytes(d);
  const size_t dkr = align_up(static_cast<size_t>(d.B) * d.skv_pad * (d.n_h / dkdv_heads_per_cta(d.n_h)) * 64 * 4, 256);
  const size_t rows = align_up(static_cast<size_t>(d.B) * d.n_h * d.sq_pad * 4, 256);
  return 4 * kv + dkr + 2 * rows;
}

BwdWorkspace tc_bwd_carve(const Dims& d, void* ws) {
  char* p = static_cast<char*>(ws);
  const size_t kv = kv_ws_bytes(d);
  BwdWorkspace w{};
  w.k_ws = reinterpret_cast<bf16*>(p);
  p += kv;
  w.v_ws = reinterpret_cast<bf16*>(p);
  p += kv;
  w.dk_ws = reinterpret_cast<bf16*>(p);
  p += kv;
  w.dv_ws = reinterpret_cast<bf16*>(p);
  p += kv;
  w.dkr_ws = reinterpret_cast<float*>(p);
  p += align_up(static_cast<size_t>(d.B) * d.skv_pad * (d.n_h / dkdv_heads_per_cta(d.n_h)) * 64 * 4, 256);
  w.lse2 = reinterpret_cast<float*>(p);
  p += align_up(static_cast<size_t>(d.B) * d.n_h * d.sq_pad * 4, 256);
  w.delta = reinterpret_cast<float*>(p);
  return w;
}

namespace {

constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ uint32_t pack_bf16x2_dev(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Half a warp per (b, h, i) row of the padded [B][n_h][sq_pad] arrays: 16 lanes
// x 8 values of out and dout each, as 16-byte loads.
__global__ void bwd_pre_kernel(Dims d, const bf16* __restrict__ out, const bf16* __restrict__ dout,
                               const float* __restrict__ lse, float* __restrict__ lse2, float* __restrict__ delta) {
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const long long rows = static_cast<long long>(d.B) * d.n_h * d.sq_pad;
  const int l16 = threadIdx.x & 15;
  const bool in = row < rows;  // every lane stays for the shuffles below
  const int i = in ? static_cast<int>(row % d.sq_pad) : 0;
  const long long bh = in ? row / d.sq_pad : 0;
  const int h = static_cast<int>(bh % d.n_h);
  const int b = static_cast<int>(bh / d.n_h);
  float acc = 0.f;
  if (in && i < d.Sq) {
    const long long off = ((static_cast<long long>(b) * d.Sq + i) * d.n_h + h) * 128 + l16 * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(out + off);
    const uint4 g = *reinterpret_cast<const uint4*>(dout + off);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 af = __bfloat1622float2(a2[k]);
      const float2 gf = __bfloat1622float2(g2[k]);
      acc = fmaf(af.x, gf.x, acc);
      acc = fmaf(af.y, gf.y, acc);
    }
  }
  for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (in && l16 == 0) {
    if (i >= d.Sq) {
      lse2[row] = INFINITY;
      delta[row] = 0.f;
    } else {
      delta[row] = acc;
      lse2[row] = lse[(static_cast<long long>(b) * d.n_h + h) * d.Sq + i] * LOG2E;
    }
  }
}

// dk_rope[b, j, :] = sum_g dkr[b, j, g, :] over the dK/dV kernel's head-group
// partials; 16 threads x 4 columns per row.
__global__ void rope_sum_kernel(Dims d, int parts, const float* __restrict__ dkr, bf16* __restrict__ dk_rope) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(d.B) * d.S * 16;
  if (t >= total) return;
  const int c4 = static_cast<int>(t % 16);
  const long long bj = t / 16;
  const int j = static_cast<int>(bj % d.S);
  const int b = static_cast<int>(bj / d.S);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (j < d.skv_pad) {
    const float4* src =
        reinterpret_cast<const float4*>(dkr + ((static_cast<long long>(b) * d.skv_pad + j) * parts) * 64) + c4;
    for (int g = 0; g < parts; ++g) {
      const float4 v = src[g * 16];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
  }
  uint2 o;
  o.x = pack_bf16x2_dev(acc.x, acc.y);
  o.y = pack_bf16x2_dev(acc.z, acc.w);
  reinterpret_cast<uint2*>(dk_rope + (static_cast<long long>(b) * d.S + j) * 64)[c4] = o;
}

}  // namespace

LaunchResult tc_bwd_pre(const Dims& d, const bf16* out, const bf16* dout, const float* lse, const BwdWorkspace& w,
                        cudaStream_t st) {
  LaunchResult r;
  const long long rows = static_cast<long long>(d.B) * d.n_h * d.sq_pad;
  bwd_pre_kernel<<<static_cast<unsigned>((rows + 15) / 16), 256, 0, st>>>(d, out, dout, lse, w.lse2, w.delta);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "bwd_pre_kernel";
  return r;
}

LaunchResult tc_bwd_post(const Dims& d, const BwdWorkspace& w, bf16* dk_rope, cudaStream_t st) {
  LaunchResult r;
  const long long t = static_cast<long long>(d.B) * d.S * 16;
  rope_sum_kernel<<<static_cast<unsigned>((t + 255) / 256), 256, 0, st>>>(d, d.n_h / dkdv_heads_per_cta(d.n_h),
                                                                          w.dkr_ws, dk_rope);
  r.err = cudaGetLastError();
  if (r.err != cudaSuccess) r.what = "bwd post kernels";
  return r;
}

}  // namespace laga
