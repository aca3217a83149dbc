/*
 * laga_mla.h — C ABI of the LAGA MLA attention block for one GPU (sm_103a).
 *
 * What the operation is
 * ---------------------
 * "A Training-Memory Regression in MLA Sequence Parallelism: Why Megatron-Core
 * Forbids Absorption, and LAGA -- a Communication-Efficient Fix" (weekinpapers
 * page, Abstract): LAGA keeps the absorbed MLA form's communication -- only the
 * compressed latent is all-gathered across the sequence-parallel (SP) group --
 * but rejects the absorb reformulation and instead rebuilds every head's K and
 * V locally from the gathered latent, then runs ordinary (explicit-form)
 * attention. The Abstract states the result is bit-identical to the explicit
 * form at SP=1. This library is that local computation on one SP rank. The
 * all-gather itself is outside it: the gathered latent is an input.
 *
 * For each batch element b, head h, local query i (absolute position
 * q_offset + i) and latent row j:
 *   K_nope[j,h,:] = c_kv[j,:] . W_UK[:, h*d_nope : (h+1)*d_nope]     (rebuild K)
 *   V[j,h,:]      = c_kv[j,:] . W_UV[:, h*d_v    : (h+1)*d_v]        (rebuild V)
 *   K_h[j]        = [K_nope[j,h,:] | k_rope[j,:]]     (one RoPE key shared by all heads)
 *   s_ij          = softmax_scale * q[i,h,:] . K_h[j], visible iff j <= q_offset+i
 *                   (causal) or always (non-causal)
 *   lse[h,i]      = ln sum_j exp(s_ij)                 over visible j
 *   out[i,h,:]    = sum_j exp(s_ij - lse[h,i]) V[j,h,:]
 * and the backward of the loss <dout, out> with respect to q, c_kv, k_rope,
 * W_UK and W_UV.
 *
 * Layouts (dense, row-major, innermost last)
 * ------------------------------------------
 *   q       [B, Sq, n_h, d_nope + d_rope]  no-RoPE part first, then RoPE part
 *   c_kv    [B, Skv, d_c]                  the gathered latent
 *   k_rope  [B, Skv, d_rope]               already rotated
 *   W_UK    [d_c, n_h * d_nope]            column h*d_nope + k belongs to head h
 *   W_UV    [d_c, n_h * d_v]               column h*d_v + k belongs to head h
 *   out     [B, Sq, n_h, d_v]
 *   lse     [B, n_h, Sq]                   always fp32, natural log of scaled scores
 *   dq, dc_kv, dk_rope, dW_UK, dW_UV       the shapes of q, c_kv, k_rope, W_UK, W_UV
 *
 * Conventions
 * -----------
 *  - Element type: every tensor has desc->dtype except lse (always fp32).
 *  - Ownership: the caller allocates every buffer, outputs and workspace
 *    included. The library allocates, frees and synchronises nothing
 *    (laga_mla_check excepted, which synchronises the given stream). All work
 *    is enqueued on the given stream (a cudaStream_t; NULL = legacy default).
 *  - Outputs are overwritten, never accumulated into.
 *  - Latent rows no query of the shard can see (j >= q_offset + Sq when causal)
 *    get zero dc_kv and dk_rope.
 *  - Alignment: every pointer 16-byte aligned. Otherwise LAGA_ERR_INVALID_ARG.
 *  - Errors: argument errors are found on the host and returned before any
 *    launch. Launch failures return LAGA_ERR_CUDA. A device-side wait that runs
 *    out (a bounded mbarrier wait) records LAGA_ERR_TIMEOUT in a per-device
 *    status word that laga_mla_check reads. No call aborts the process.
 *  - Threads: calls are re-entrant as long as concurrent calls use disjoint
 *    workspaces and outputs.
 *  - Reproducibility: no kernel uses atomics; every output is produced in a
 *    fixed order, so repeated calls give bitwise-identical results.
 *  - Device resets: the library caches, per device and CUDA context, the device
 *    addresses of its module globals (the status word, the static scratch of
 *    laga_mla_fwd_noalloc); a new context after cudaDeviceReset is detected and
 *    the addresses are looked up again. Calls must not run while another thread
 *    resets the device.
 *
 * Supported problems
 * ------------------
 *  - dtype BF16 with d_c = 512, d_nope = d_v = 128, d_rope = 64 (the
 *    DeepSeek-V3 dimensions): tensor-core path (tcgen05/TMEM/TMA).
 *  - dtype F32, any dims with d_nope + d_rope <= 256, d_v <= 256, d_c <= 1024:
 *    CUDA-core path in fp32 (also available for BF16 via LAGA_VARIANT_SIMT).
 *  - batch, Sq, Skv >= 1, n_h >= 1, 0 <= q_offset, and q_offset + Sq <= Skv
 *    when causal.
 */
#ifndef LAGA_MLA_H
#define LAGA_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t. */
typedef struct CUstream_st* laga_stream_t;

typedef enum {
  LAGA_OK = 0,
  LAGA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad sizes, q_offset+Sq > Skv when causal */
  LAGA_ERR_UNSUPPORTED = 2, /* sizes or dtype this build has no kernel for */
  LAGA_ERR_WORKSPACE = 3,   /* workspace pointer null or smaller than the query function said */
  LAGA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or kernel launch failed */
  LAGA_ERR_TIMEOUT = 5      /* a device-side bounded wait expired (reported by laga_mla_check) */
} laga_status;

typedef enum { LAGA_DTYPE_F32 = 0, LAGA_DTYPE_BF16 = 1 } laga_dtype;

/* How K and V reach the attention kernels.
 *  MATERIALIZE: one tensor-core GEMM writes every head's K_nope and V to the
 *               workspace in HBM, the attention kernels read them back.
 *  FUSED_RECON: forward only — each attention CTA rebuilds its K_nope/V tiles
 *               from the latent tile on the tensor cores, nothing is written.
 *  SIMT:        the fp32 CUDA-core kernels (any dims).
 *  AUTO:        MATERIALIZE for the supported BF16 dims, else SIMT. */
typedef enum {
  LAGA_VARIANT_AUTO = 0,
  LAGA_VARIANT_MATERIALIZE = 1,
  LAGA_VARIANT_FUSED_RECON = 2,
  LAGA_VARIANT_SIMT = 3
} laga_variant;

typedef struct {
  int64_t batch;     /* B */
  int64_t sq;        /* local query rows of this SP rank */
  int64_t skv;       /* gathered latent length S */
  int64_t n_h;       /* heads */
  int64_t d_c;       /* latent width */
  int64_t d_nope;    /* per-head no-RoPE query/key width */
  int64_t d_rope;    /* RoPE query/key width (key shared by all heads) */
  int64_t d_v;       /* per-head value width */
  int64_t q_offset;  /* absolute position of local query row 0 */
  int32_t causal;    /* nonzero: key j visible to local query i iff j <= q_offset + i */
  float softmax_scale; /* <= 0 selects 1/sqrt(d_nope + d_rope) */
  int32_t dtype;     /* laga_dtype */
  int32_t variant;   /* laga_variant */
  int32_t flags;     /* bitwise OR of laga_flags (0 = none) */
  /* Two-segment query shard (zigzag sequence parallelism: rank r holds chunks r and
   * 2*SP-1-r of the sequence, which evens out the causal work across ranks).
   * q_split = 0: one segment, rows i at q_offset + i (q_offset2 ignored).
   * 0 < q_split < sq: rows i < q_split sit at q_offset + i, rows i >= q_split at
   * q_offset2 + (i - q_split). q_split must be a multiple of 128, and the call must
   * take the tensor-core materialize path (bf16, the supported dims; AUTO picks it).
   * Causal shards need q_offset + q_split <= skv and q_offset2 + sq - q_split <= skv. */
  int64_t q_split;
  int64_t q_offset2;
} laga_mla_desc;

/* Descriptor flags.
 *  LAGA_FLAG_REUSE_KV (laga_mla_bwd): the workspace passed to laga_mla_bwd is
 *    the one laga_mla_fwd used for the same inputs and descriptor, and its
 *    first laga_mla_fwd_workspace_size bytes still hold the per-head K_nope
 *    and V the forward rebuilt there. The backward then reads them instead of
 *    rebuilding them. The backward workspace layout starts with the forward
 *    one, so one buffer of laga_mla_bwd_workspace_size bytes serves both
 *    calls. Keeping K/V alive between the calls is the memory profile of the
 *    explicit MLA form, which stores per-head K and V for its backward. */
/*  LAGA_FLAG_KV_PREBUILT (laga_mla_fwd): the workspace already holds this call's
 *    per-head K_nope and V for every latent row the forward reads, written there
 *    by laga_mla_reconstruct_rows with the same descriptor (in any number of row
 *    ranges, in any order, on this stream or on one ordered before it). The
 *    forward then runs the attention alone. A sequence-parallel caller can so
 *    rebuild each chunk of the gathered latent as soon as that chunk has
 *    arrived, overlapping the rebuild with the rest of the gather (the Abstract's
 *    LAGA gathers the latent and rebuilds K/V locally). Tensor-core materialize
 *    path only (LAGA_ERR_UNSUPPORTED otherwise). */
typedef enum { LAGA_FLAG_REUSE_KV = 1, LAGA_FLAG_KV_PREBUILT = 2 } laga_flags;

/* Bytes of device workspace laga_mla_fwd / laga_mla_bwd need for this
 * problem (0 if the descriptor is invalid or unsupported). The workspace must
 * be 256-byte aligned and must not be shared by calls in flight. */
size_t laga_mla_fwd_workspace_size(const laga_mla_desc* desc);
size_t laga_mla_bwd_workspace_size(const laga_mla_desc* desc);

/* Forward of the attention block on one SP rank: out [B,Sq,n_h,d_v] (dtype) and
 * lse [B,n_h,Sq] (fp32).
 * Source: the LAGA page's Abstract (weekinpapers, "A Training-Memory Regression in
 * MLA Sequence Parallelism ..."): each rank rebuilds every head's K and V from the
 * gathered latent instead of absorbing W_UK into the query, then runs the
 * explicit form's attention, whose result LAGA reproduces exactly at SP=1. The
 * RoPE-key concat and the causal rule at the shard's offset are as defined at the
 * top of this file.
 * Arguments: q, c_kv, k_rope, W_UK, W_UV are read-only inputs in the layouts
 * above; out and lse are written in full; workspace is caller-owned scratch of at
 * least laga_mla_fwd_workspace_size bytes (256-byte aligned) that the call
 * overwrites. All pointers are device pointers. Errors: LAGA_ERR_INVALID_ARG /
 * UNSUPPORTED / WORKSPACE before any launch, LAGA_ERR_CUDA if a launch fails. */
laga_status laga_mla_fwd(const laga_mla_desc* desc, const void* q, const void* c_kv, const void* k_rope,
                         const void* W_UK, const void* W_UV, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, laga_stream_t stream);

/* Backward of the attention block for the loss <dout, out>: the gradients a
 * training step needs (the Abstract's setting is MLA training under sequence
 * parallelism), through the attention and through the local K/V rebuild.
 * Source: the LAGA page's Abstract, as for laga_mla_fwd; the softmax gradient is
 * the textbook one (dS = P o (dP - rowsum(dout o out))).
 * Arguments: out and lse are the forward's outputs for the same inputs and
 * descriptor; dout has out's shape. Writes dq, dc_kv, dk_rope, dW_UK, dW_UV in
 * full (all dtype, shapes of their primals; dW sums over the batch; dc_kv and
 * dk_rope are this rank's partial sums, which an SP group adds up). workspace:
 * at least laga_mla_bwd_workspace_size bytes, 256-byte aligned, overwritten
 * (see LAGA_FLAG_REUSE_KV for sharing it with the forward). All pointers are
 * device pointers. Errors as for laga_mla_fwd. */
laga_status laga_mla_bwd(const laga_mla_desc* desc, const void* q, const void* c_kv, const void* k_rope,
                         const void* W_UK, const void* W_UV, const void* out, const float* lse,
                         const void* dout, void* dq, void* dc_kv, void* dk_rope, void* dW_UK, void* dW_UV,
                         void* workspace, size_t workspace_bytes, laga_stream_t stream);

/* Step 1 alone, LAGA's local K/V rebuild (the LAGA page's Abstract: per-head K
 * and V are reconstructed on each rank from the gathered latent):
 * k_nope [B,Skv,n_h,d_nope] = c_kv . W_UK and v [B,Skv,n_h,d_v] = c_kv . W_UV,
 * per head, for all Skv rows, written in full. Device pointers; needs no
 * workspace; only the descriptor's batch, skv, n_h, d_c, d_nope, d_v, dtype and
 * variant are used. Errors as for laga_mla_fwd. */
laga_status laga_mla_reconstruct(const laga_mla_desc* desc, const void* c_kv, const void* W_UK,
                                 const void* W_UV, void* k_nope, void* v, laga_stream_t stream);

/* laga_mla_fwd's step 1 (the local K/V rebuild) for latent rows [row0, row0 + rows)
 * of every batch element, into the forward workspace, for a later laga_mla_fwd
 * with LAGA_FLAG_KV_PREBUILT and the same descriptor. The forward reads the rows
 * of the padded visible prefix, [0, Skv_pad) with Skv_pad the last row any query
 * sees plus one, rounded up to 128; the calls must cover it, and rows past it are
 * ignored. row0 must be a multiple of 128 and row0 + rows either a multiple of
 * 128 or at least Skv_pad. c_kv, W_UK, W_UV are the full device tensors of
 * laga_mla_fwd; workspace and workspace_bytes as for laga_mla_fwd (its contents
 * outside the rebuilt rows are left alone). Tensor-core materialize path only.
 * Errors: LAGA_ERR_INVALID_ARG (range), LAGA_ERR_UNSUPPORTED (path),
 * LAGA_ERR_WORKSPACE before any launch; LAGA_ERR_CUDA if the launch fails. */
laga_status laga_mla_reconstruct_rows(const laga_mla_desc* desc, const void* c_kv, const void* W_UK,
                                      const void* W_UV, int64_t row0, int64_t rows, void* workspace,
                                      size_t workspace_bytes, laga_stream_t stream);

/* The absorbed MLA form, forward, for comparison with the library's own path.
 * Source: the LAGA page's Abstract (weekinpapers, "A Training-Memory Regression
 * in MLA Sequence Parallelism ..."): Megatron-Core's absorbed form folds W_UK
 * into the query and attends over the compressed latent itself; LAGA keeps its
 * latent-only communication but rejects the reformulation because of the
 * memory its intermediates take. Per head h:
 *   q_lat  = q_nope_h . W_UK_h^T                         [B, Sq, d_c]
 *   s_ij   = softmax_scale * ([q_lat | q_rope]_i . [c_kv | k_rope]_j)  (masked as above)
 *   ctx_i  = sum_j softmax_j(s_ij) c_kv_j                [B, Sq, d_c]
 *   out_i  = ctx_i . W_UV_h
 * The scores are the explicit form's, so out and lse equal laga_mla_fwd's up to
 * rounding. The intermediates q_lat and ctx (n_h * d_c values per query row
 * each) live in the workspace: laga_mla_absorbed_fwd_workspace_size bytes,
 * 256-byte aligned. Supported: bf16 with the tensor-core dims, one query
 * segment, variant AUTO. Arguments, layouts and errors as for laga_mla_fwd. */
size_t laga_mla_absorbed_fwd_workspace_size(const laga_mla_desc* desc);
laga_status laga_mla_absorbed_fwd(const laga_mla_desc* desc, const void* q, const void* c_kv, const void* k_rope,
                                  const void* W_UK, const void* W_UV, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, laga_stream_t stream);

/* Largest workspace, in bytes, that laga_mla_fwd_noalloc can stand in for. */
#define LAGA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* Forward for callers that cannot allocate device memory, and so have no
 * workspace to pass: a plug-in whose host framework owns all device memory
 * through its own pool, a runtime with a fixed memory budget, a C caller
 * without an allocator. Same arguments and results as laga_mla_fwd minus the
 * workspace; the caller still passes every input and output. The paper has no
 * counterpart of this entry point: it exists for those callers only.
 *
 * The forward's scratch (the per-head K_nope and V) lives in one static device
 * array of LAGA_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits. Problems whose laga_mla_fwd_workspace_size exceeds
 * it return LAGA_ERR_WORKSPACE (laga_mla_last_error says by how much). The
 * first call on each device looks up the array's device address (set-up done
 * once per device, with that device current); make that first call before any
 * stream capture. Every call on a device shares the array, which keeps the last
 * call's contents; calls whose kernels overlap on the GPU race on it, so
 * serialise them. Allocates nothing: no cudaMalloc, cudaFree or allocating
 * library routine. */
laga_status laga_mla_fwd_noalloc(const laga_mla_desc* desc, const void* q, const void* c_kv, const void* k_rope,
                                 const void* W_UK, const void* W_UV, void* out, float* lse, laga_stream_t stream);

/* Synchronises the stream, then reads and clears this device's status word.
 * Returns LAGA_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last
 * check, LAGA_ERR_CUDA if the stream reports an error, else LAGA_OK. */
laga_status laga_mla_check(laga_stream_t stream);

/* Static string naming a status code. */
const char* laga_status_string(laga_status status);

/* Detail of the last error returned on this host thread (static storage). */
const char* laga_mla_last_error(void);

/* Optional kernel timing. While enabled on the calling host thread, each step
 * that laga_mla_fwd / laga_mla_bwd launch (one kernel, or a short group of
 * memory-bound kernels named after their role) is bracketed by two CUDA
 * events recorded on the caller's stream. Enabling (or
 * disabling) clears earlier records. The events are created on first use and
 * reused; nothing is recorded while disabled (the default). */
laga_status laga_mla_profile_enable(int enable);

/* Waits for the recorded events and writes, for up to `max` launches in launch
 * order, the kernel's name (static string) and its elapsed time in ms.
 * Returns the number of launches recorded since the last enable (which may
 * exceed `max`), or -1 if an event query fails. */
int laga_mla_profile_read(const char** names, float* ms, int max);

/* Failure-path self test. Enqueues on `stream` one CTA whose thread waits on an
 * mbarrier that nothing ever arrives at, through the same bounded wait every
 * library kernel uses (2 s, wait site 99). The wait expires, the kernel records
 * LAGA_ERR_TIMEOUT in this device's status word exactly as a library kernel that
 * gave up on a wait does, and returns; the CUDA context stays usable. The next
 * laga_mla_check on the stream then returns LAGA_ERR_TIMEOUT (and clears the
 * word). Returns LAGA_ERR_CUDA if the launch fails, else LAGA_OK. */
laga_status laga_mla_selftest_timeout(laga_stream_t stream);

/* Library ABI version: major*10000 + minor*100 + patch. 200 (0.2.0): laga_mla_desc
 * gained q_split and q_offset2 (two-segment query shards); zero them for the
 * single-segment behaviour of 100. */
int laga_mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LAGA_MLA_H */
