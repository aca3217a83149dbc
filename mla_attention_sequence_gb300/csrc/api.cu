// C ABI of the LAGA MLA attention block: argument validation, workspace
// layout, dispatch between the tensor-core and CUDA-core kernels, status
// reporting. Nothing here allocates device memory.
#include "../../include/laga_mla.h"
#include "internal.h"
#include "ptx.cuh"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

namespace laga {

__device__ int g_device_status = 0;

namespace {

thread_local char t_last_error[512] = "";

laga_status fail(laga_status s, const char* fmt, const char* detail = nullptr) {
  std::snprintf(t_last_error, sizeof(t_last_error), fmt, detail ? detail : "");
  return s;
}

laga_status from_launch(const LaunchResult& r) {
  if (r.ok()) return LAGA_OK;
  if (r.err != cudaSuccess) {
    std::snprintf(t_last_error, sizeof(t_last_error), "%s: %s", r.what ? r.what : "CUDA", cudaGetErrorString(r.err));
  } else {
    std::snprintf(t_last_error, sizeof(t_last_error), "%s: CUresult %d", r.what ? r.what : "driver",
                  static_cast<int>(r.cu));
  }
  return LAGA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- opt-in kernel timing: one event pair per launch, events pooled per thread.
// Each record keeps the pool indices of its own two events, so a launch whose
// events could not be created is skipped without shifting the pairs after it.
struct ProfRecord {
  const char* name;
  size_t begin, end;  // indices into pool
};
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  std::vector<ProfRecord> recs;
  size_t used = 0;  // events handed out since the last enable
  bool open = false;  // a begin was recorded and awaits its end
};
thread_local Profiler t_prof;

// Index of the next free pooled event (created on first use), or -1.
long prof_event() {
  Profiler& P = t_prof;
  if (P.used == P.pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return -1;
    P.pool.push_back(e);
  }
  return static_cast<long>(P.used++);
}

// Records the start event of a launch named `name` (no-op when disabled).
void prof_begin(const char* name, cudaStream_t s) {
  Profiler& P = t_prof;
  P.open = false;
  if (!P.on) return;
  const long e = prof_event();
  if (e < 0 || cudaEventRecord(P.pool[e], s) != cudaSuccess) return;
  P.recs.push_back(ProfRecord{name, static_cast<size_t>(e), 0});
  P.open = true;
}

void prof_end(cudaStream_t s) {
  Profiler& P = t_prof;
  if (!P.on || !P.open) return;
  P.open = false;
  const long e = prof_event();
  if (e < 0 || cudaEventRecord(P.pool[e], s) != cudaSuccess) {
    P.recs.pop_back();  // no end event: drop the record
    return;
  }
  P.recs.back().end = static_cast<size_t>(e);
}

// Run one launcher between two profiling marks.
template <class F>
LaunchResult timed(const char* name, cudaStream_t s, F&& f) {
  prof_begin(name, s);
  LaunchResult r = f();
  prof_end(s);
  return r;
}

enum class Path { Invalid, Simt, TensorCore, TensorCoreFused };

// Validate the descriptor; fill dims; choose a path. On error, sets *st.
Path plan(const laga_mla_desc* desc, Dims* d, laga_status* st, bool for_bwd) {
  *st = LAGA_OK;
  if (!desc) {
    *st = fail(LAGA_ERR_INVALID_ARG, "null descriptor%s");
    return Path::Invalid;
  }
  const laga_mla_desc& x = *desc;
  if (x.batch < 1 || x.sq < 1 || x.skv < 1 || x.n_h < 1 || x.d_c < 1 || x.d_nope < 1 || x.d_rope < 0 || x.d_v < 1 ||
      x.q_offset < 0) {
    *st = fail(LAGA_ERR_INVALID_ARG, "sizes must be positive (d_rope >= 0, q_offset >= 0)%s");
    return Path::Invalid;
  }
  // Bound every factor first, so that the products below cannot overflow.
  const int64_t lim = int64_t(1) << 30;
  if (x.skv >= lim || x.sq >= lim || x.q_offset >= lim || (x.q_split != 0 && x.q_offset2 >= lim) ||
      x.batch >= 65536 ||
      x.n_h >= 65536 || x.d_c >= 65536 || x.d_nope >= 65536 || x.d_rope >= 65536 || x.d_v >= 65536) {
    *st = fail(LAGA_ERR_UNSUPPORTED, "problem too large%s");
    return Path::Invalid;
  }
  if (x.batch * x.skv * x.n_h * (x.d_nope + x.d_rope + x.d_v) >= (int64_t(1) << 40) ||
      x.batch * x.sq * x.n_h * (x.d_nope + x.d_rope + x.d_v) >= (int64_t(1) << 40)) {
    *st = fail(LAGA_ERR_UNSUPPORTED, "problem too large%s");
    return Path::Invalid;
  }
  const bool two_seg = x.q_split != 0;
  if (two_seg && (x.q_split < 0 || x.q_split >= x.sq || x.q_split % 128 != 0 || x.q_offset2 < 0)) {
    *st = fail(LAGA_ERR_INVALID_ARG, "q_split must be 0 or a multiple of 128 in (0, sq), q_offset2 >= 0%s");
    return Path::Invalid;
  }
  if (x.causal && x.q_offset + (two_seg ? x.q_split : x.sq) > x.skv) {
    *st = fail(LAGA_ERR_INVALID_ARG, "causal shard needs q_offset + sq <= skv%s");
    return Path::Invalid;
  }
  if (x.causal && two_seg && x.q_offset2 + (x.sq - x.q_split) > x.skv) {
    *st = fail(LAGA_ERR_INVALID_ARG, "causal shard needs q_offset2 + sq - q_split <= skv%s");
    return Path::Invalid;
  }
  if ((x.flags & ~static_cast<int32_t>(LAGA_FLAG_REUSE_KV | LAGA_FLAG_KV_PREBUILT)) != 0) {
    *st = fail(LAGA_ERR_INVALID_ARG, "unknown bits in flags%s");
    return Path::Invalid;
  }
  if (x.dtype != LAGA_DTYPE_F32 && x.dtype != LAGA_DTYPE_BF16) {
    *st = fail(LAGA_ERR_UNSUPPORTED, "dtype must be LAGA_DTYPE_F32 or LAGA_DTYPE_BF16%s");
    return Path::Invalid;
  }
  d->B = static_cast<int>(x.batch);
  d->Sq = static_cast<int>(x.sq);
  d->S = static_cast<int>(x.skv);
  d->n_h = static_cast<int>(x.n_h);
  d->d_c = static_cast<int>(x.d_c);
  d->d_nope = static_cast<int>(x.d_nope);
  d->d_rope = static_cast<int>(x.d_rope);
  d->d_v = static_cast<int>(x.d_v);
  d->q_offset = static_cast<int>(x.q_offset);
  d->q_split = two_seg ? static_cast<int>(x.q_split) : 0;
  d->q_offset2 = two_seg ? static_cast<int>(x.q_offset2) : 0;
  d->causal = x.causal != 0;
  d->scale = x.softmax_scale > 0.f ? x.softmax_scale : 1.0f / std::sqrt(static_cast<float>(x.d_nope + x.d_rope));
  // latent rows any query can see: the furthest position of either segment, plus one
  d->skv_eff = d->causal ? (two_seg ? std::max(d->q_offset + d->q_split, d->q_offset2 + d->Sq - d->q_split)
                                    : d->q_offset + d->Sq)
                         : d->S;
  d->skv_pad = static_cast<int>(align_up(static_cast<size_t>(d->skv_eff), 128));
  d->sq_pad = static_cast<int>(align_up(static_cast<size_t>(d->Sq), 128));

  const bool want_simt = x.variant == LAGA_VARIANT_SIMT;
  const bool tc_ok = x.dtype == LAGA_DTYPE_BF16 && tc_supported(*d);
  if (x.variant < LAGA_VARIANT_AUTO || x.variant > LAGA_VARIANT_SIMT) {
    *st = fail(LAGA_ERR_INVALID_ARG, "unknown variant%s");
    return Path::Invalid;
  }
  if (!want_simt && x.variant != LAGA_VARIANT_AUTO && !tc_ok) {
    *st = fail(LAGA_ERR_UNSUPPORTED,
               "tensor-core variants need bf16 with d_c=512, d_nope=d_v=128, d_rope=64%s");
    return Path::Invalid;
  }
  if (two_seg && (want_simt || !tc_ok || x.variant == LAGA_VARIANT_FUSED_RECON)) {
    *st = fail(LAGA_ERR_UNSUPPORTED, "two query segments need the tensor-core materialize path%s");
    return Path::Invalid;
  }
  if (x.variant == LAGA_VARIANT_FUSED_RECON) {
    if (for_bwd) {
      *st = fail(LAGA_ERR_UNSUPPORTED, "LAGA_VARIANT_FUSED_RECON is forward-only%s");
      return Path::Invalid;
    }
    return Path::TensorCoreFused;
  }
  if (tc_ok && !want_simt) return Path::TensorCore;
  // CUDA-core path limits (shared-memory rows of scores).
  if (x.d_nope + x.d_rope > 1024 || x.d_v > 1024 || x.skv > 49152 || x.sq > 24576) {
    *st = fail(LAGA_ERR_UNSUPPORTED, "CUDA-core path supports skv <= 49152, sq <= 24576%s");
    return Path::Invalid;
  }
  return Path::Simt;
}

using CuTensorMapEncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                            const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                            CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                            CUtensorMapFloatOOBfill);

CuTensorMapEncodeTiled encode_fn() {
  static CuTensorMapEncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CuTensorMapEncodeTiled>(p);
  });
  return fn;
}


using CuCtxGetCurrent = CUresult (*)(CUcontext*);

CuCtxGetCurrent ctx_fn() {
  static CuCtxGetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CuCtxGetCurrent>(p);
  });
  return fn;
}

}  // namespace

void set_last_error(const char* msg) { std::snprintf(t_last_error, sizeof(t_last_error), "%s", msg); }

int sm_count() {
  static int counts[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    counts[dev] = n;
  }
  return counts[dev];
}

void* current_context() {
  CuCtxGetCurrent fn = ctx_fn();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

int* device_status_ptr() {
  // Cached per device together with the context it was looked up in: a new
  // primary context (after cudaDeviceReset) reloads the module, and the word
  // may then sit at another address.
  static int* ptrs[64] = {};
  static void* ctxs[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev] || ctxs[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
    ctxs[dev] = ctx;
  }
  return ptrs[dev];
}

CUresult make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  CuTensorMapEncodeTiled fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  return fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides_bytes, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// One thread waits on an mbarrier nothing arrives at; the bounded wait expires
// and the timeout lands in the status word like any kernel's expired wait.
__global__ void selftest_timeout_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int* abort_flag = &abort_word;
    if (!mbar_wait_or_abort(&bar, 0, abort_flag, 99)) publish_abort(abort_flag, status);
  }
}

}  // namespace laga

using namespace laga;

extern "C" {

size_t laga_mla_fwd_workspace_size(const laga_mla_desc* desc) {
  Dims d{};
  laga_status st;
  switch (plan(desc, &d, &st, false)) {
    case Path::Simt: return simt_fwd_workspace(d);
    case Path::TensorCore: return tc_fwd_workspace(d);
    case Path::TensorCoreFused: return 0;
    default: return 0;
  }
}

size_t laga_mla_bwd_workspace_size(const laga_mla_desc* desc) {
  Dims d{};
  laga_status st;
  switch (plan(desc, &d, &st, true)) {
    case Path::Simt: return simt_bwd_workspace(d);
    case Path::TensorCore: return tc_bwd_workspace(d);
    default: return 0;
  }
}

laga_status laga_mla_fwd(const laga_mla_desc* desc, const void* q, const void* c_kv, const void* k_rope,
                         const void* W_UK, const void* W_UV, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, laga_stream_t stream) {
  Dims d{};
  laga_status st;
  const Path path = plan(desc, &d, &st, false);
  if (path == Path::Invalid) return st;
  const void* ptrs[] = {q, c_kv, W_UK, W_UV, out, lse};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(LAGA_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned%s");
  if (d.d_rope > 0 && (!k_rope || !aligned16(k_rope)))
    return fail(LAGA_ERR_INVALID_ARG, "k_rope must be non-null and 16-byte aligned%s");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = desc->dtype == LAGA_DTYPE_BF16;
  if ((desc->flags & LAGA_FLAG_KV_PREBUILT) && path != Path::TensorCore)
    return fail(LAGA_ERR_UNSUPPORTED, "LAGA_FLAG_KV_PREBUILT needs the tensor-core materialize path%s");
  if (path == Path::TensorCoreFused) {
    return from_launch(timed("attn_fwd_fused", s, [&] {
      return tc_attn_fwd_fused(d, static_cast<const bf16*>(q), static_cast<const bf16*>(c_kv),
                               static_cast<const bf16*>(W_UK), static_cast<const bf16*>(W_UV),
                               static_cast<const bf16*>(k_rope), static_cast<bf16*>(out), lse, s);
    }));
  }
  const size_t need = path == Path::Simt ? simt_fwd_workspace(d) : tc_fwd_workspace(d);
  if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return fail(LAGA_ERR_WORKSPACE, "workspace missing, misaligned (256 B) or too small%s");
  if (path == Path::Simt)
    return from_launch(
        timed("simt_fwd", s, [&] { return simt_fwd(d, bf, q, c_kv, k_rope, W_UK, W_UV, out, lse, workspace, s); }));
  bf16* k_ws = static_cast<bf16*>(workspace);
  bf16* v_ws = k_ws + static_cast<size_t>(d.B) * d.skv_pad * d.n_h * 128;
  if (!(desc->flags & LAGA_FLAG_KV_PREBUILT)) {
    LaunchResult r = timed("recon_fwd_gemm", s, [&] {
      return tc_recon_fwd(d, static_cast<const bf16*>(c_kv), static_cast<const bf16*>(W_UK),
                          static_cast<const bf16*>(W_UV), k_ws, v_ws, d.skv_pad, s);
    });
    if (!r.ok()) return from_launch(r);
  }
  return from_launch(timed("attn_fwd", s, [&] {
    return tc_attn_fwd(d, static_cast<const bf16*>(q), k_ws, v_ws, static_cast<const bf16*>(k_rope),
                       static_cast<bf16*>(out), lse, s);
  }));
}

laga_status laga_mla_reconstruct_rows(const laga_mla_desc* desc, const void* c_kv, const void* W_UK,
                                      const void* W_UV, int64_t row0, int64_t rows, void* workspace,
                                      size_t workspace_bytes, laga_stream_t stream) {
  Dims d{};
  laga_status st;
  const Path path = plan(desc, &d, &st, false);
  if (path == Path::Invalid) return st;
  if (path != Path::TensorCore)
    return fail(LAGA_ERR_UNSUPPORTED, "laga_mla_reconstruct_rows needs the tensor-core materialize path%s");
  const void* ptrs[] = {c_kv, W_UK, W_UV};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(LAGA_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned%s");
  if (row0 < 0 || rows <= 0 || row0 % 128 != 0 || row0 > (int64_t{1} << 40) || rows > (int64_t{1} << 40))
    return fail(LAGA_ERR_INVALID_ARG, "row0 must be a non-negative multiple of 128 and rows positive%s");
  const int64_t end = std::min<int64_t>(row0 + rows, d.skv_pad);
  if (row0 >= d.skv_pad) return LAGA_OK;  // rows no query sees: nothing to rebuild
  if (end % 128 != 0) return fail(LAGA_ERR_INVALID_ARG, "row0 + rows must be a multiple of 128 or reach Skv_pad%s");
  const size_t need = tc_fwd_workspace(d);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LAGA_ERR_WORKSPACE, "workspace missing, misaligned (256 B) or too small%s");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bf16* k_ws = static_cast<bf16*>(workspace);
  bf16* v_ws = k_ws + static_cast<size_t>(d.B) * d.skv_pad * d.n_h * 128;
  return from_launch(timed("recon_fwd_gemm", s, [&] {
    return tc_recon_fwd(d, static_cast<const bf16*>(c_kv), static_cast<const bf16*>(W_UK),
                        static_cast<const bf16*>(W_UV), k_ws, v_ws, d.skv_pad, s, static_cast<int>(row0 / 128),
                        static_cast<int>((end - row0) / 128));
  }));
}

laga_status laga_mla_bwd(const laga_mla_desc* desc, const void* q, const void* c_kv, const void* k_rope,
                         const void* W_UK, const void* W_UV, const void* out, const float* lse, const void* dout,
                         void* dq, void* dc_kv, void* dk_rope, void* dW_UK, void* dW_UV, void* workspace,
                         size_t workspace_bytes, laga_stream_t stream) {
  Dims d{};
  laga_status st;
  const Path path = plan(desc, &d, &st, true);
  if (path == Path::Invalid) return st;
  const void* ptrs[] = {q, c_kv, W_UK, W_UV, out, lse, dout, dq, dc_kv, dW_UK, dW_UV};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(LAGA_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned%s");
  if (d.d_rope > 0 && (!k_rope || !aligned16(k_rope) || !dk_rope || !aligned16(dk_rope)))
    return fail(LAGA_ERR_INVALID_ARG, "k_rope/dk_rope must be non-null and 16-byte aligned%s");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = desc->dtype == LAGA_DTYPE_BF16;
  const size_t need = path == Path::Simt ? simt_bwd_workspace(d) : tc_bwd_workspace(d);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LAGA_ERR_WORKSPACE, "workspace missing, misaligned (256 B) or too small%s");
  if (path == Path::Simt)
    return from_launch(timed("simt_bwd", s, [&] {
      return simt_bwd(d, bf, q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, dq, dc_kv, dk_rope, dW_UK, dW_UV,
                      workspace, (desc->flags & LAGA_FLAG_REUSE_KV) != 0, s);
    }));
  BwdWorkspace w = tc_bwd_carve(d, workspace);
  auto cb = [](const void* p) { return static_cast<const bf16*>(p); };
  LaunchResult r;
  if (!(desc->flags & LAGA_FLAG_REUSE_KV))
    r = timed("recon_fwd_gemm", s,
              [&] { return tc_recon_fwd(d, cb(c_kv), cb(W_UK), cb(W_UV), w.k_ws, w.v_ws, d.skv_pad, s); });
  if (r.ok()) r = timed("bwd_pre", s, [&] { return tc_bwd_pre(d, cb(out), cb(dout), lse, w, s); });
  if (r.ok())
    r = timed("attn_bwd_dkdv", s, [&] { return tc_attn_bwd_dkdv(d, cb(q), cb(k_rope), cb(dout), w, s); });
  if (r.ok())
    r = timed("attn_bwd_dq", s,
              [&] { return tc_attn_bwd_dq(d, cb(q), cb(k_rope), cb(dout), w, static_cast<bf16*>(dq), s); });
  if (r.ok())
    r = timed("recon_bwd_dc_gemm", s, [&] {
      return tc_recon_bwd_dc(d, w.dk_ws, w.dv_ws, cb(W_UK), cb(W_UV), static_cast<bf16*>(dc_kv), s);
    });
  if (r.ok())
    r = timed("recon_bwd_dw_gemm", s, [&] {
      return tc_recon_bwd_dw(d, cb(c_kv), w.dk_ws, w.dv_ws, static_cast<bf16*>(dW_UK), static_cast<bf16*>(dW_UV), s);
    });
  if (r.ok())
    r = timed("bwd_post", s, [&] { return tc_bwd_post(d, w, static_cast<bf16*>(dk_rope), s); });
  if (r.ok() && d.skv_pad < d.S) {
    // Latent rows beyond the padded visible prefix get zero gradient.
    r.err = cudaMemset2DAsync(static_cast<bf16*>(dc_kv) + static_cast<size_t>(d.skv_pad) * d.d_c,
                              static_cast<size_t>(d.S) * d.d_c * 2, 0, static_cast<size_t>(d.S - d.skv_pad) * d.d_c * 2,
                              d.B, s);
    if (r.err != cudaSuccess) r.what = "zero dc_kv tail";
  }
  return from_launch(r);
}

laga_status laga_mla_reconstruct(const laga_mla_desc* desc, const void* c_kv, const void* W_UK, const void* W_UV,
                                 void* k_nope, void* v, laga_stream_t stream) {
  Dims d{};
  laga_status st;
  const Path path = plan(desc, &d, &st, false);
  if (path == Path::Invalid) return st;
  const void* ptrs[] = {c_kv, W_UK, W_UV, k_nope, v};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(LAGA_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned%s");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (path == Path::TensorCore || path == Path::TensorCoreFused) {
    // The GEMM writes whole 128-row tiles; full tiles go straight to the
    // output, and a ragged tail is computed by the CUDA-core kernel.
    const int full = d.S / 128 * 128;
    LaunchResult r;
    if (full > 0) {
      Dims dd = d;
      // Batch stride of the output is S rows: write per batch element.
      for (int b = 0; b < d.B && r.ok(); ++b) {
        dd.B = 1;
        const bf16* cb = static_cast<const bf16*>(c_kv) + static_cast<size_t>(b) * d.S * d.d_c;
        bf16* kb = static_cast<bf16*>(k_nope) + static_cast<size_t>(b) * d.S * d.n_h * 128;
        bf16* vb = static_cast<bf16*>(v) + static_cast<size_t>(b) * d.S * d.n_h * 128;
        dd.S = full;
        r = tc_recon_fwd(dd, cb, static_cast<const bf16*>(W_UK), static_cast<const bf16*>(W_UV), kb, vb, full, s);
      }
    }
    if (r.ok() && full < d.S) {
      for (int b = 0; b < d.B && r.ok(); ++b) {
        Dims dt = d;
        dt.B = 1;
        dt.S = d.S - full;
        const bf16* cb = static_cast<const bf16*>(c_kv) + (static_cast<size_t>(b) * d.S + full) * d.d_c;
        bf16* kb = static_cast<bf16*>(k_nope) + (static_cast<size_t>(b) * d.S + full) * d.n_h * 128;
        bf16* vb = static_cast<bf16*>(v) + (static_cast<size_t>(b) * d.S + full) * d.n_h * 128;
        r = simt_reconstruct(dt, true, cb, W_UK, W_UV, kb, vb, false, s);
      }
    }
    return from_launch(r);
  }
  const bool bf = desc->dtype == LAGA_DTYPE_BF16;
  return from_launch(simt_reconstruct(d, bf, c_kv, W_UK, W_UV, k_nope, v, !bf, s));
}

size_t laga_mla_absorbed_fwd_workspace_size(const laga_mla_desc* desc) {
  Dims d{};
  laga_status st;
  if (plan(desc, &d, &st, false) != Path::TensorCore || d.q_split > 0) return 0;
  const size_t lat = align_up(static_cast<size_t>(d.B) * d.Sq * d.n_h * d.d_c * 2, 256);
  return 2 * lat;  // q_lat and the latent-space context
}

laga_status laga_mla_absorbed_fwd(const laga_mla_desc* desc, const void* q, const void* c_kv, const void* k_rope,
                                  const void* W_UK, const void* W_UV, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, laga_stream_t stream) {
  Dims d{};
  laga_status st;
  const Path path = plan(desc, &d, &st, false);
  if (path == Path::Invalid) return st;
  if (path != Path::TensorCore || d.q_split > 0 || desc->variant != LAGA_VARIANT_AUTO)
    return fail(LAGA_ERR_UNSUPPORTED,
                "the absorbed form runs for bf16 with d_c=512, d_nope=d_v=128, d_rope=64, one query segment%s");
  const void* ptrs[] = {q, c_kv, k_rope, W_UK, W_UV, out, lse};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return fail(LAGA_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned%s");
  const size_t lat = align_up(static_cast<size_t>(d.B) * d.Sq * d.n_h * d.d_c * 2, 256);
  if (!workspace || workspace_bytes < 2 * lat || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LAGA_ERR_WORKSPACE, "workspace missing, misaligned (256 B) or too small%s");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bf16* q_lat = static_cast<bf16*>(workspace);
  bf16* ctx = reinterpret_cast<bf16*>(static_cast<char*>(workspace) + lat);
  auto cb = [](const void* ptr) { return static_cast<const bf16*>(ptr); };
  LaunchResult r = timed("absorbed_qlat_gemm", s, [&] { return tc_absorbed_qlat(d, cb(q), cb(W_UK), q_lat, s); });
  if (r.ok())
    r = timed("absorbed_attn", s,
              [&] { return tc_absorbed_attn(d, q_lat, cb(q), cb(c_kv), cb(k_rope), ctx, lse, s); });
  if (r.ok())
    r = timed("absorbed_out_gemm", s,
              [&] { return tc_absorbed_outproj(d, ctx, cb(W_UV), static_cast<bf16*>(out), s); });
  return from_launch(r);
}

laga_status laga_mla_selftest_timeout(laga_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* status = device_status_ptr();
  if (status == nullptr) {
    std::snprintf(t_last_error, sizeof(t_last_error), "device status word unavailable");
    return LAGA_ERR_CUDA;
  }
  selftest_timeout_kernel<<<1, 32, 0, s>>>(status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    std::snprintf(t_last_error, sizeof(t_last_error), "selftest launch: %s", cudaGetErrorString(e));
    return LAGA_ERR_CUDA;
  }
  return LAGA_OK;
}

laga_status laga_mla_check(laga_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    std::snprintf(t_last_error, sizeof(t_last_error), "stream: %s", cudaGetErrorString(e));
    return LAGA_ERR_CUDA;
  }
  int status = 0;
  const int zero = 0;
  e = cudaMemcpyFromSymbolAsync(&status, g_device_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && status != 0)
    e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    std::snprintf(t_last_error, sizeof(t_last_error), "status word: %s", cudaGetErrorString(e));
    return LAGA_ERR_CUDA;
  }
  if ((status & 0xff) == kStatusTimeout) {
    std::snprintf(t_last_error, sizeof(t_last_error), "device wait expired (site %d)", status >> 8);
    return LAGA_ERR_TIMEOUT;
  }
  return LAGA_OK;
}

const char* laga_status_string(laga_status status) {
  switch (status) {
    case LAGA_OK: return "LAGA_OK";
    case LAGA_ERR_INVALID_ARG: return "LAGA_ERR_INVALID_ARG";
    case LAGA_ERR_UNSUPPORTED: return "LAGA_ERR_UNSUPPORTED";
    case LAGA_ERR_WORKSPACE: return "LAGA_ERR_WORKSPACE";
    case LAGA_ERR_CUDA: return "LAGA_ERR_CUDA";
    case LAGA_ERR_TIMEOUT: return "LAGA_ERR_TIMEOUT";
  }
  return "LAGA_ERR_UNKNOWN";
}

const char* laga_mla_last_error(void) { return t_last_error; }

laga_status laga_mla_profile_enable(int enable) {
  t_prof.on = enable != 0;
  t_prof.used = 0;
  t_prof.open = false;
  t_prof.recs.clear();
  return LAGA_OK;
}

int laga_mla_profile_read(const char** names, float* ms, int max) {
  const Profiler& P = t_prof;
  const int n = static_cast<int>(P.recs.size());
  for (int i = 0; i < n && i < max; ++i) {
    const ProfRecord& r = P.recs[i];
    if (cudaEventSynchronize(P.pool[r.end]) != cudaSuccess) return -1;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, P.pool[r.begin], P.pool[r.end]) != cudaSuccess) return -1;
    if (names) names[i] = r.name;
    if (ms) ms[i] = t;
  }
  return n;
}

int laga_mla_version(void) { return 200; }

}  // extern "C"
