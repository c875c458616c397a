// smla_internal.cuh -- declarations shared by the CUDA translation units of
// libsmla.so (device helpers, workspace carving, kernel launchers).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/smla.h"

namespace smla {

constexpr int kD = 512;                 // head width fixed by the contract
constexpr int kWarp = 32;

// ---------------------------------------------------------------- status word
// The first 256 bytes of every workspace hold a status word: bit `code` is
// set when a kernel meets the condition of that code (SMLA_ERR_INDEX,
// SMLA_ERR_TIMEOUT). The host clears it at the start of each call.
constexpr size_t kStatusBytes = 256;

// Byte 64 of the status area: the work counter of the S/dP/dS kernel's
// dynamic item scheduling, zeroed on the stream before each launch.
inline int* sdi_work_counter(unsigned* status) {
    return reinterpret_cast<int*>(reinterpret_cast<char*>(status) + 64);
}

__device__ __forceinline__ void flag_status(unsigned* status, int code) {
    atomicOr(status, 1u << code);
}

// Reads topk[t, r] and classifies it: returns the row index, or -1 for a
// masked slot. Indices outside [-1, num_kv) are reported and treated as masked.
__device__ __forceinline__ int load_index(const int32_t* p, int num_kv, unsigned* status) {
    int j = __ldg(p);
    if (j < -1 || j >= num_kv) {
        flag_status(status, SMLA_ERR_INDEX);
        j = -1;
    }
    return j;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Two floats -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Returns SMLA_OK if every non-NULL pointer of `ptrs` is device memory of the
// current device (or managed memory), else SMLA_ERR_DEVICE (SMLA_ERR_CUDA if
// the device cannot be queried).
int check_device_ptrs(const void* const* ptrs, int n);

// ------------------------------------------------------------ workspace plans
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The scale*dS^T stash of the tensor-core path is [T, Rp, Hp] bf16: ranks padded
// to whole 128-rank tiles, heads padded to whole 64-column swizzle blocks.
inline int round_up_ranks(int R) { return (R + 127) / 128 * 128; }
inline int pad_heads(int H) { return H <= 64 ? 64 : 128; }

// Radix-sort based CSR build parameters.
constexpr int kRadixBits = 11;
constexpr int kRadixBuckets = 1 << kRadixBits;   // 2048
constexpr int kRadixWarps = 8;
constexpr int kRadixPerWarp = 1024;
constexpr int kRadixBlock = kRadixWarps * kRadixPerWarp;  // entries per radix block

// dKV gather: a kv row's contributor list is cut into segments of at most
// kGatherSeg entries; each segment is summed on its own and the segments of a
// row are then added in order.
constexpr int kGatherSeg = 256;

struct CsrPlan {
    int64_t n;          // entries T * r_len
    int nblk;           // radix blocks
    int passes;         // radix passes
    int64_t nscan;      // counters per pass (buckets * nblk)
    size_t off_keys0, off_vals0, off_keys1, off_vals1, off_cnt, off_scan_tmp;
    size_t bytes;       // scratch bytes (excluding row_ptr / col)
};

CsrPlan plan_csr(int64_t T, int64_t r_len, int64_t num_kv);

struct BwdPlan {
    int64_t T, H, K, N, R;   // R = rank chunk
    int nchunks;
    bool full_stash;         // chunked, R a multiple of 128: one dS^T stash of all ranks
    bool compact;            // unchunked: the kernels read a compacted index table (below)
    CsrPlan csr;
    int64_t max_segs;
    size_t off_delta, off_rowptr, off_col, off_csr, off_segptr, off_segrow, off_segcnt,
        off_scan_tmp2, off_partial, off_interm, off_dst, off_dqacc, off_dkvacc, off_cidx, off_ccnt;
    size_t bytes;
};

BwdPlan plan_bwd(const smla_dims& d);

// Scratch of the generic exclusive scan (int32) over n values.
size_t scan_tmp_bytes(int64_t n);

// ------------------------------------------------------- launch accounting
// Every launcher calls note_launch() once per kernel it enqueues; the phase
// profiler attributes the count to the running phase.
void note_launch(int n = 1);

// ---------------------------------------------------------------- launchers
// All launchers enqueue on `s` and return cudaGetLastError().
cudaError_t launch_delta(const uint16_t* o, const uint16_t* dO, float* delta,
                         int64_t rows, cudaStream_t s);
cudaError_t launch_dsink(const float* delta, const float* lse, const float* sink,
                         float* d_sink, int T, int H, cudaStream_t s);
// out[i] = partials[0][i] + partials[1][i] + ... + partials[n_parts-1][i], added
// in that order in fp32 (n a multiple of 4); bf16 (RNE) and / or fp32 outputs.
cudaError_t launch_reduce_partials(const float* partials, int n_parts, int64_t n,
                                   uint16_t* out_bf16, float* out_f32, cudaStream_t s);
cudaError_t launch_exclusive_scan(const int32_t* in, int32_t* out, int64_t n,
                                  void* tmp, cudaStream_t s, bool write_total);
// Compacted index table: row t of `cidx` [T, K] holds the valid entries of
// topk row t (0 <= j < num_kv), in rank order, then -1; cnt[t] = their number.
// Indices outside [-1, num_kv) set SMLA_ERR_INDEX and count as masked.
cudaError_t launch_compact_ranks(const int32_t* topk, int T, int K, int num_kv, int32_t* cidx,
                                 int32_t* cnt, unsigned* status, cudaStream_t s);
cudaError_t launch_csr(const int32_t* topk, int T, int topk_w, int r0, int r_len, int num_kv,
                       int32_t* row_ptr, int32_t* col, char* scratch, const CsrPlan& p,
                       unsigned* status, cudaStream_t s);
cudaError_t launch_gather(const int32_t* row_ptr, const int32_t* col, const uint16_t* interm,
                          int num_kv, int64_t max_segs, int32_t* seg_cnt, int32_t* seg_ptr,
                          int32_t* seg_row, void* scan_tmp, float* partial, float* dkv_acc,
                          uint16_t* dkv_out, bool first_chunk, bool last_chunk, cudaStream_t s);
cudaError_t launch_fwd(const uint16_t* q, const uint16_t* kv, const int32_t* topk,
                       const float* sink, uint16_t* o, float* lse, int T, int H, int K,
                       int num_kv, float scale, unsigned* status, cudaStream_t s);
// Tensor-core forward (H a multiple of 32 up to 128, 1 <= topk <= 512); returns
// cudaErrorNotSupported for other shapes. launch_fwd tries it first.
cudaError_t launch_fwd_tc(const uint16_t* q, const uint16_t* kv, const int32_t* topk,
                          const float* sink, uint16_t* o, float* lse, int T, int H, int K,
                          int num_kv, float scale, unsigned* status, cudaStream_t s);

// Per-chunk attention backward core: for ranks [r0, r0+R) of each token, builds
// interm [T, R, D] bf16 (sum_h P*dO + scale*dS*q) and the scale*dS^T stash
// (bf16, heads padded to Hp), then accumulates dq. The stash has ds_rows rank
// rows per token and the chunk's rows start at ds_off: round_up(R, 128) and 0
// for a stash of the chunk alone, or topk and r0 for one stash of all ranks
// (then dq runs once over all ranks, after the last chunk).
struct ChunkArgs {
    const uint16_t* q; const uint16_t* kv; const uint16_t* dO;
    const float* lse; const float* delta; const int32_t* topk;
    // with `cnt` set, topk is a compacted table (valid entries first, then -1)
    // and cnt[t] the number of valid entries of token t
    const int32_t* cnt;
    int T, H, K, N, r0, R;
    float scale;
    uint16_t* interm; uint16_t* dsT;
    int ds_rows, ds_off;
    float* dq_acc; uint16_t* dq_out;   // dq_acc NULL when unchunked
    bool first_chunk, last_chunk;
    // dq runs beside only part of the dKV gather (rank chunks): it gets more SMs
    bool dq_beside_part;
    unsigned* status;
};
// The two tensor-core kernels of one chunk: S/dP/P/dS + interm (+ dS stash),
// then dq from the stash. launch_attn_dq must follow launch_attn_sdi.
cudaError_t launch_attn_sdi(const ChunkArgs& a, cudaStream_t s);
// One CTA whose bounded mbarrier wait (limit_ns) runs out on purpose: sets
// SMLA_ERR_TIMEOUT in `status` through the kernels' own unwind path.
cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_attn_dq(const ChunkArgs& a, cudaStream_t s);

}  // namespace smla
