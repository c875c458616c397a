/*
 * smla.h -- C ABI of the GB300 (sm_103a) sparse MLA attention library.
 *
 * The operation is the DeepSeek-V4 sparse MLA attention of the aiter pull
 * request "[WIP][TRITON][GLUON][GFX950][DSV4] Sparse MLA training backward":
 *
 *   Contract section: shared-KV GQA with K == V == kv, one dense bf16
 *   [num_kv, 512] tensor; scale 1/sqrt(512); a per-head attn_sink folded into
 *   the softmax denominator only; topk_indices == -1 masked out; num_kv >= T
 *   allowed, so rows T..num_kv-1 can be a compressed pool. The forward's lse
 *   is sink-inclusive: lse = e_max + log(e_sum) with the sink folded in.
 *
 *   Usage example in that section: o, lse = forward(q, kv, topk, sink) and
 *   dq, dkv, d_sink = backward(q, kv, do, o, lse, topk, sink). This header
 *   exports the same two calls (smla_fwd, smla_bwd), plus the inverted top-k
 *   CSR build of the Structure section (smla_csr_build).
 *
 * Conventions (all entry points):
 *   - Every tensor is a row-major, contiguous DEVICE buffer owned by the
 *     caller (HOST buffers for smla_bwd_host): q, dO, o, dq are [T, H, D];
 *     kv, dkv are [num_kv, D]; lse is [T, H]; topk is [T, topk]; sink, d_sink
 *     are [H]. bf16 tensors are passed as uint16_t bit patterns.
 *   - Every device pointer must be 16-byte aligned, and must point to device
 *     (or managed) memory of the current device: each is checked with
 *     cudaPointerGetAttributes before anything is enqueued (SMLA_ERR_DEVICE).
 *     The library cannot see how long a caller's buffer is: each must hold
 *     the tensor that the shape says.
 *   - The library allocates no device memory during a call. The caller passes
 *     a device workspace of at least smla_workspace_size() bytes. Between calls
 *     the library keeps a per-device cache of the arch check and, per host
 *     thread and device, the streams and events it creates on first use: a
 *     side stream on which smla_bwd builds the CSR (forked from and joined back
 *     into `stream` with events) and the two copy streams of smla_bwd_host.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously. A returned SMLA_OK means the work was
 *     launched, not that it finished.
 *   - Host-side validation happens before any launch: on an error code
 *     nothing was enqueued and no output was touched.
 *   - An index in topk outside [-1, num_kv) is never dereferenced: it is
 *     treated as masked and the kernel sets SMLA_ERR_INDEX in a status word
 *     inside the workspace; read it with smla_get_device_status().
 *   - Results are deterministic: the same inputs give bitwise identical
 *     outputs on every run (no floating-point atomics anywhere).
 */
#ifndef SMLA_H
#define SMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point (and found in the device status word). */
enum smla_status {
    SMLA_OK = 0,
    SMLA_ERR_NULL = 1,          /* a required pointer is NULL */
    SMLA_ERR_SHAPE = 2,         /* T/H/topk/num_kv out of the supported range */
    SMLA_ERR_D512 = 3,          /* D != 512 (the contract fixes the width) */
    SMLA_ERR_NUM_KV_LT_T = 4,   /* num_kv < T */
    SMLA_ERR_RCHUNK = 5,        /* r_chunk does not divide topk */
    SMLA_ERR_ALIGN = 6,         /* a pointer is not 16-byte aligned */
    SMLA_ERR_OVERLAP = 7,       /* an output overlaps an input, another output or the workspace */
    SMLA_ERR_WORKSPACE = 8,     /* workspace NULL or smaller than smla_workspace_size() */
    SMLA_ERR_ARCH = 9,          /* current device is not compute capability 10.3 (sm_103) */
    SMLA_ERR_CUDA = 10,         /* a CUDA runtime call failed */
    SMLA_ERR_INDEX = 11,        /* device: a topk entry outside [-1, num_kv) was seen */
    SMLA_ERR_TIMEOUT = 12,      /* device: a bounded wait inside a kernel ran out */
    SMLA_ERR_SINK = 13,         /* d_sink given without sink, or sink without d_sink */
    SMLA_ERR_ARG = 14,          /* any other invalid argument (e.g. a non-finite scale) */
    SMLA_ERR_DEVICE = 15        /* a pointer that must be device memory is not device (or managed)
                                   memory of the current device */
};

/* Problem dimensions. */
typedef struct smla_dims {
    int32_t T;        /* query tokens */
    int32_t H;        /* query heads sharing the one kv tensor: a multiple of 16, 16..128 */
    int32_t D;        /* head width: must be 512 */
    int32_t topk;     /* ranks per token (columns of topk) */
    int32_t num_kv;   /* rows of kv (>= T; rows >= T are the compressed pool) */
    int32_t r_chunk;  /* backward rank chunk: 0 = topk (unchunked); else must divide topk */
    float scale;      /* score scale: 0 = 1/sqrt(D) */
} smla_dims;

/* Operation selector for smla_workspace_size. */
enum smla_op { SMLA_OP_FWD = 0, SMLA_OP_BWD = 1, SMLA_OP_CSR = 2, SMLA_OP_BWD_HOST = 3 };

/*
 * Workspace bytes needed by one call of `op` with these dimensions
 * (SMLA_OP_BWD_HOST: smla_bwd_host, the backward's workspace plus device
 * copies of its inputs and outputs).
 * For SMLA_OP_CSR the fields used are T, topk (the row width of the index
 * table), r_chunk (the number of ranks covered, 0 = topk) and num_kv.
 * Returns SMLA_OK and writes *bytes, or a validation error.
 */
int smla_workspace_size(int op, const smla_dims* dims, size_t* bytes);

/*
 * Sparse MLA forward (the has_pe=False prefill forward the page composes with:
 * its usage example, and the lse convention under it).
 * For each token t and head h, over the valid ranks r (topk[t,r] != -1):
 *   s_r = scale * <q[t,h,:], kv[topk[t,r],:]>
 *   lse[t,h] = log(exp(sink[h]) + sum_r exp(s_r))      (natural log; no sink term if sink == NULL)
 *   o[t,h,:] = sum_r exp(s_r - lse[t,h]) * kv[topk[t,r],:]
 * A row with no valid rank gets o = 0 and lse = sink[h] (or -inf without a sink).
 *   q [T,H,D] bf16, kv [num_kv,D] bf16, topk [T,topk] int32, sink [H] fp32 or NULL
 *   -> o [T,H,D] bf16 (round to nearest even), lse [T,H] fp32.
 * Kernels: for H a multiple of 32 and topk <= 512, a tensor-core kernel
 * (S and O on tcgen05). It rounds exp(s_r - m) (m = the row max, sink
 * included) to bf16 as the operand of the O product and divides the fp32
 * result by the fp32 row sum before rounding o to bf16. Other shapes use a
 * CUDA-core kernel with fp32 weights.
 */
int smla_fwd(const uint16_t* q, const uint16_t* kv, const int32_t* topk,
             const float* sink, uint16_t* o, float* lse,
             const smla_dims* dims, void* workspace, size_t workspace_bytes,
             void* stream);

/*
 * Sparse MLA training backward (the Structure section's delta, dQ,
 * dKV-interm, CSR build, atomic-free dKV gather and d_sink phases).
 * With P = exp(s - lse) rebuilt from the GIVEN lse and delta from the GIVEN o:
 *   delta[t,h]  = sum_d o[t,h,d] * dO[t,h,d]
 *   dS[t,h,r]   = P * (<dO[t,h,:], kv[idx_r,:]> - delta[t,h])
 *   dq[t,h,:]   = scale * sum_r dS * kv[idx_r,:]
 *   dkv[j,:]    = sum over (t,h,r) with idx_r = j of  P * dO[t,h,:] + scale * dS * q[t,h,:]
 *   d_sink[h]   = -sum_t exp(sink[h] - lse[t,h]) * delta[t,h]
 *   inputs : q, dO, o [T,H,D] bf16; kv [num_kv,D] bf16; lse [T,H] fp32 (sink-inclusive);
 *            topk [T,topk] int32; sink [H] fp32 or NULL
 *   outputs: dq [T,H,D] bf16; dkv [num_kv,D] bf16; d_sink [H] fp32 (NULL iff sink is NULL)
 * dims->r_chunk splits the ranks into chunks processed in order (the page's
 * R_CHUNK): it bounds the workspace; dq and dkv are accumulated in fp32
 * across chunks and rounded to bf16 once.
 * T == 0 is allowed: dkv is zeroed and d_sink is zeroed.
 */
int smla_bwd(const uint16_t* q, const uint16_t* kv, const uint16_t* dO,
             const uint16_t* o, const float* lse, const int32_t* topk,
             const float* sink, uint16_t* dq, uint16_t* dkv, float* d_sink,
             const smla_dims* dims, void* workspace, size_t workspace_bytes,
             void* stream);

/*
 * One rank's share of a token-sharded backward (several GPUs, each holding a
 * slice of the tokens; the RL-Kernel page's "Algorithmic arrangements" item 5:
 * partials combined in a fixed rank order, the collective used only to move
 * them). Same arguments, layouts and errors as smla_bwd for the rank's T
 * tokens, except the kv gradient and d_sink are left as fp32 partial sums over
 * these tokens, unrounded:
 *   dkv_partial [num_kv, D] fp32 = sum over this rank's (t, h, r) of the dkv terms;
 *   d_sink_partial [H] fp32 (NULL iff sink is NULL) = -sum over this rank's t of
 *   exp(sink - lse) * delta.
 * dq of the rank's tokens is final (bf16). Every rank passes the full kv and
 * gathers the others' partials; smla_reduce_partials then adds them in rank
 * order and rounds once.
 */
int smla_bwd_partial(const uint16_t* q, const uint16_t* kv, const uint16_t* dO,
                     const uint16_t* o, const float* lse, const int32_t* topk,
                     const float* sink, uint16_t* dq, float* dkv_partial,
                     float* d_sink_partial, const smla_dims* dims, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Ordered sum of n_parts partials (the combine step of a token-sharded
 * backward): for every i in [0, n),
 *   s = partials[0][i] + partials[1][i] + ... + partials[n_parts - 1][i]
 * added left to right in fp32, so every rank that runs it on the same gathered
 * partials gets the same bits. Writes s rounded to bf16 (RNE) to out_bf16
 * and / or s to out_f32 (either may be NULL, not both).
 *   partials [n_parts, n] fp32 (contiguous, device); n a multiple of 4.
 * Errors: SMLA_ERR_NULL, SMLA_ERR_SHAPE (n_parts < 1, n < 0 or not a
 * multiple of 4), SMLA_ERR_ALIGN, SMLA_ERR_OVERLAP, SMLA_ERR_DEVICE.
 */
int smla_reduce_partials(const float* partials, int32_t n_parts, int64_t n,
                         uint16_t* out_bf16, float* out_f32, void* stream);

/*
 * The same backward with every input and output in HOST memory (the pages
 * have no such call; it is the end-to-end form of smla_bwd). Arguments,
 * results and errors are those of smla_bwd, except that q, kv, dO, o, lse,
 * topk, sink, dq, dkv and d_sink are host pointers (no alignment rule), and the
 * workspace (device memory, 16-byte aligned) must hold
 * smla_workspace_size(SMLA_OP_BWD_HOST) bytes: the backward's own workspace
 * followed by device copies of the inputs and outputs.
 * The call enqueues work and returns: host-to-device copies run on an internal
 * copy stream, small inputs first (the CSR build needs only topk), then o, dO
 * and q in chunks of about 512 tokens; each token chunk's delta, S/dP/dS and dq
 * start as soon as its inputs have arrived, while later chunks are still
 * being copied; each chunk's dq goes back to the host on a second copy stream
 * as soon as it is final, then dkv and d_sink. `stream` waits for all of it:
 * the host outputs are valid once `stream` (or an event recorded on it after
 * the call) has completed. Host buffers must stay valid and unchanged until
 * then. Use page-locked host memory (cudaHostAlloc / cudaHostRegister) for the
 * copies to run asynchronously; pageable memory also works, with copies that
 * do not overlap.
 */
int smla_bwd_host(const uint16_t* q, const uint16_t* kv, const uint16_t* dO,
                  const uint16_t* o, const float* lse, const int32_t* topk,
                  const float* sink, uint16_t* dq, uint16_t* dkv, float* d_sink,
                  const smla_dims* dims, void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * Inverted top-k CSR over the ranks [r0, r0 + r_len) of each row of topk
 * (the Structure section's CSR build; the page uses sort + searchsorted).
 * With p = t * r_len + (r - r0), the flat position in a [T, r_len, D]
 * intermediate:
 *   row_ptr[j]                      = number of valid entries with index < j
 *   col[row_ptr[j] .. row_ptr[j+1]) = every p with topk[t, r] == j, ascending
 * -1 entries are dropped; nnz = row_ptr[num_kv] <= T * r_len.
 *   topk [T, topk_w] int32 -> row_ptr [num_kv + 1] int32, col [T * r_len] int32
 *   (entries of col at and beyond nnz are left unspecified).
 * The result is unique and bit-exact. Requires 0 <= r0, r_len >= 1,
 * r0 + r_len <= topk_w, num_kv >= 1.
 */
int smla_csr_build(const int32_t* topk, int32_t T, int32_t topk_w, int32_t r0,
                   int32_t r_len, int32_t num_kv, int32_t* row_ptr, int32_t* col,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * d_sink without a workspace. The page has no counterpart to this entry point:
 * it exists for callers that cannot allocate device memory -- because another
 * allocator (a framework's caching allocator, or an arena reserved at
 * start-up) owns all of it, or because they run where allocating is not
 * allowed -- and so cannot hand smla_bwd a workspace. It computes the same
 * d_sink as smla_bwd, with the same kernels:
 *   delta[t,h] = sum_d o[t,h,d] * dO[t,h,d];  d_sink[h] = -sum_t exp(sink[h] - lse[t,h]) * delta[t,h]
 *   dO, o [T,H,D=512] bf16; lse [T,H] fp32; sink [H] fp32 -> d_sink [H] fp32 (all device memory).
 * The scratch (delta) lives in a 4 MiB array inside the library, so the call
 * allocates nothing. Limits and rules:
 *   - T * H must be <= 1048576 (2^20), else SMLA_ERR_SHAPE and nothing runs;
 *     H must be a multiple of 16 in 16..128.
 *   - The array exists on every GPU that loads the library, until the process exits.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. The address belongs to the device's current
 *     CUDA context: after cudaDeviceReset the first call in the new context
 *     looks it up again (same rule).
 *   - All calls share the array: calls whose kernels overlap on the GPU race,
 *     so serialize them (one stream, or events between streams).
 */
int smla_dsink_static(const uint16_t* dO, const uint16_t* o, const float* lse,
                      const float* sink, float* d_sink, int32_t T, int32_t H, void* stream);

/*
 * Self-test of the kernels' bounded waits (the pages have no counterpart; it
 * exists so that the failure path can be exercised without faulting a GPU).
 * Launches one CTA that waits on an mbarrier nothing arrives on, through the
 * same wait-and-unwind code as the tensor-core kernels, with a limit of
 * `limit_us` microseconds (1 .. 1000000): the wait runs out, the CTA sets
 * SMLA_ERR_TIMEOUT in the workspace's status word, stops its other warps,
 * frees its tensor memory and exits. Read the result with
 * smla_get_device_status(); the device stays usable afterwards.
 *   workspace: device memory of at least 256 bytes (its status word is reset).
 */
int smla_selftest_wait_timeout(void* workspace, size_t workspace_bytes, uint32_t limit_us,
                               void* stream);

/*
 * Synchronizes `stream`, then reads the device status word that the last
 * call given this workspace wrote (SMLA_OK, SMLA_ERR_INDEX or
 * SMLA_ERR_TIMEOUT) into *status. Returns SMLA_ERR_CUDA if the stream or
 * the copy failed.
 */
int smla_get_device_status(const void* workspace, void* stream, int* status);

/*
 * Phase profiling (tracing aid; off by default). While enabled, smla_bwd
 * brackets each of its phases with CUDA events on the stream that runs it (the
 * caller's; the CSR build runs on the library's side stream, overlapped with
 * the others, so its span is not its own run time) and counts the kernels it
 * launches. The aiter page reports a per-kernel sum
 * next to the end-to-end time (Performance table); these counters give the
 * same split.
 *   smla_profiling(1) enables and resets; smla_profiling(0) disables.
 *   smla_profile_read() synchronizes on every pending event, then writes up to
 *   `max` phase records to `out` and their count to *n. Phase names are
 *   static strings. Not thread-safe: profile from one host thread.
 */
typedef struct smla_phase_stat {
    const char* name;      /* phase name, e.g. "delta", "csr", "attn", "gather", "dsink" */
    double total_ms;       /* summed event time of the phase */
    long long calls;       /* times the phase ran */
    long long launches;    /* kernels launched by the phase */
} smla_phase_stat;

int smla_profiling(int enable);
int smla_profile_read(smla_phase_stat* out, int max, int* n);

/* Static, human-readable text for a status code. Never NULL. */
const char* smla_status_string(int code);

/* Library ABI version (major * 100 + minor). */
int smla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SMLA_H */
