// k_csr.cu -- inverted top-k CSR build on the GPU.
//
// The aiter page ("Sparse MLA training backward", Structure table, CSR build)
// inverts the rank -> kv-row scatter into per-kv-row contributor lists with
// torch sort + searchsorted on int16-narrowed keys. Here the same CSR is built
// by a stable LSD radix sort of (key = kv row, value = flat position p) pairs,
// whose input is already in ascending p order; a stable sort therefore leaves
// each row's positions ascending, which makes the CSR unique (bit-exact).
// Keys are full int32 (no narrowing); masked slots get the sentinel key
// num_kv and sort past every real row, so nnz = row_ptr[num_kv].
//
// Each pass over 11 key bits is three kernels: per-block digit histograms,
// an exclusive scan over (digit, block), and a stable scatter in which each
// warp walks its 1024 entries in order and ranks equal digits with
// __match_any_sync. Work and scratch are O(T * r_len + num_kv): nothing is
// sized by T * num_kv.
#include "smla_internal.cuh"

namespace smla {

struct KeySource {
    const int32_t* keys;   // NULL: read pass-0 keys from the top-k table
    const int32_t* vals;
    const int32_t* topk;
    int topk_w, r0, r_len, num_kv;
    unsigned* status;
};

__device__ __forceinline__ void load_entry(const KeySource& src, int64_t e, int& key, int& val) {
    if (src.keys) {
        key = src.keys[e];
        val = src.vals[e];
    } else {
        const int64_t t = e / src.r_len;
        const int r = int(e - t * src.r_len);
        const int j = load_index(src.topk + t * src.topk_w + src.r0 + r, src.num_kv, src.status);
        key = j < 0 ? src.num_kv : j;
        val = int(e);
    }
}

// One warp per token row, in batches of 512 entries: each lane loads its 16
// entries of the batch first (independent loads, one memory latency per
// batch), then 16 ballots of the valid ones give each its place among the
// row's valid entries so far.
__global__ void __launch_bounds__(256) compact_ranks_kernel(const int32_t* __restrict__ topk, int T, int K,
                                                             int num_kv, int32_t* __restrict__ cidx,
                                                             int32_t* __restrict__ cnt, unsigned* status) {
    const int lane = threadIdx.x & 31;
    const int t = int((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    if (t >= T) return;
    const int32_t* row = topk + int64_t(t) * K;
    int32_t* out = cidx + int64_t(t) * K;
    const unsigned lt = (1u << lane) - 1u;
    int base = 0;
    for (int b0 = 0; b0 < K; b0 += 512) {
        int j[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int r = b0 + 32 * k + lane;
            j[k] = r < K ? __ldg(row + r) : -1;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (j[k] < -1 || j[k] >= num_kv) {
                flag_status(status, SMLA_ERR_INDEX);
                j[k] = -1;
            }
            const unsigned v = __ballot_sync(0xffffffffu, j[k] >= 0);
            if (j[k] >= 0) out[base + __popc(v & lt)] = j[k];
            base += __popc(v);
        }
    }
    for (int r = base + lane; r < K; r += 32) out[r] = -1;
    if (lane == 0) cnt[t] = base;
}

cudaError_t launch_compact_ranks(const int32_t* topk, int T, int K, int num_kv, int32_t* cidx,
                                 int32_t* cnt, unsigned* status, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int64_t blocks = (int64_t(T) + 7) / 8;     // 8 warps, one per token
    compact_ranks_kernel<<<unsigned(blocks), 256, 0, s>>>(topk, T, K, num_kv, cidx, cnt, status);
    note_launch();
    return cudaGetLastError();
}

CsrPlan plan_csr(int64_t T, int64_t r_len, int64_t num_kv) {
    CsrPlan p{};
    p.n = T * r_len;
    p.nblk = int((p.n + kRadixBlock - 1) / kRadixBlock);
    int bits = 1;
    while ((int64_t(1) << bits) <= num_kv) ++bits;          // sentinel num_kv must fit
    p.passes = (bits + kRadixBits - 1) / kRadixBits;
    p.nscan = int64_t(kRadixBuckets) * (p.nblk > 0 ? p.nblk : 1);
    size_t off = 0;
    const size_t nb = align_up(size_t(p.n > 0 ? p.n : 1) * 4, 256);
    p.off_keys0 = off; off += nb;
    p.off_vals0 = off; off += nb;
    p.off_keys1 = off; off += nb;
    p.off_vals1 = off; off += nb;
    p.off_cnt = off; off += align_up(size_t(p.nscan) * 4, 256);
    p.off_scan_tmp = off; off += scan_tmp_bytes(p.nscan);
    p.bytes = off;
    return p;
}

__global__ void __launch_bounds__(256) radix_hist(KeySource src, int64_t n, int shift, int nblk,
                                                  int32_t* __restrict__ cnt) {
    __shared__ int hist[kRadixBuckets];
    for (int d = threadIdx.x; d < kRadixBuckets; d += blockDim.x) hist[d] = 0;
    __syncthreads();
    const int64_t base = int64_t(blockIdx.x) * kRadixBlock;
    for (int i = threadIdx.x; i < kRadixBlock; i += blockDim.x) {
        const int64_t e = base + i;
        if (e >= n) break;
        int key, val;
        load_entry(src, e, key, val);
        atomicAdd(&hist[(key >> shift) & (kRadixBuckets - 1)], 1);
    }
    __syncthreads();
    for (int d = threadIdx.x; d < kRadixBuckets; d += blockDim.x)
        cnt[int64_t(d) * nblk + blockIdx.x] = hist[d];
}

__global__ void __launch_bounds__(kRadixWarps * 32) radix_scatter(KeySource src, int64_t n, int shift,
                                                                  int nblk,
                                                                  const int32_t* __restrict__ offs,
                                                                  int32_t* __restrict__ keys_out,
                                                                  int32_t* __restrict__ vals_out) {
    extern __shared__ int wh[];                      // [kRadixWarps][kRadixBuckets]
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int* mine = wh + w * kRadixBuckets;
    const int64_t begin = int64_t(blockIdx.x) * kRadixBlock + int64_t(w) * kRadixPerWarp;
    const int64_t end = begin + kRadixPerWarp < n ? begin + kRadixPerWarp : n;
    for (int d = lane; d < kRadixBuckets; d += 32) mine[d] = 0;
    __syncwarp();
    for (int64_t e = begin + lane; e < end; e += 32) {
        int key, val;
        load_entry(src, e, key, val);
        atomicAdd(&mine[(key >> shift) & (kRadixBuckets - 1)], 1);
    }
    __syncthreads();
    // Warp w's entries of digit d follow those of warps < w in this block and
    // those of earlier blocks (offs is scanned digit-major, block-minor).
    for (int d = threadIdx.x; d < kRadixBuckets; d += blockDim.x) {
        int run = offs[int64_t(d) * nblk + blockIdx.x];
        for (int ww = 0; ww < kRadixWarps; ++ww) {
            const int c = wh[ww * kRadixBuckets + d];
            wh[ww * kRadixBuckets + d] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t b = begin; b < end; b += 32) {
        const int64_t e = b + lane;
        const bool active = e < end;
        int key = 0, val = 0;
        if (active) load_entry(src, e, key, val);
        const int digit = active ? ((key >> shift) & (kRadixBuckets - 1)) : (kRadixBuckets + lane);
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        const int rank = __popc(peers & lt);
        if (active) {
            const int pos = mine[digit] + rank;
            keys_out[pos] = key;
            vals_out[pos] = val;
        }
        __syncwarp();
        if (active && rank == 0) mine[digit] += __popc(peers);
        __syncwarp();
    }
}

// row_ptr from the sorted keys: entries [row_ptr[j], row_ptr[j+1]) have key j.
__global__ void __launch_bounds__(256) csr_rowptr(const int32_t* __restrict__ keys, int64_t n,
                                                  int num_kv, int32_t* __restrict__ row_ptr) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i > n) return;
    const int kprev = i == 0 ? -1 : keys[i - 1];
    int k = i == n ? num_kv : keys[i];
    if (k > num_kv) k = num_kv;
    for (int j = kprev + 1; j <= k; ++j) row_ptr[j] = int(i);
}

cudaError_t launch_csr(const int32_t* topk, int T, int topk_w, int r0, int r_len, int num_kv,
                       int32_t* row_ptr, int32_t* col, char* scratch, const CsrPlan& p,
                       unsigned* status, cudaStream_t s) {
    if (p.n == 0) return cudaMemsetAsync(row_ptr, 0, sizeof(int32_t) * (size_t(num_kv) + 1), s);
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    const int smem = kRadixWarps * kRadixBuckets * int(sizeof(int));
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(radix_scatter,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int32_t* keys[2] = {reinterpret_cast<int32_t*>(scratch + p.off_keys0),
                        reinterpret_cast<int32_t*>(scratch + p.off_keys1)};
    int32_t* vals[2] = {reinterpret_cast<int32_t*>(scratch + p.off_vals0),
                        reinterpret_cast<int32_t*>(scratch + p.off_vals1)};
    int32_t* cnt = reinterpret_cast<int32_t*>(scratch + p.off_cnt);
    void* tmp = scratch + p.off_scan_tmp;
    KeySource src{nullptr, nullptr, topk, topk_w, r0, r_len, num_kv, status};
    int32_t* last_keys = nullptr;
    for (int pass = 0; pass < p.passes; ++pass) {
        const int shift = pass * kRadixBits;
        const bool final_pass = pass == p.passes - 1;
        int32_t* ko = keys[pass & 1];
        int32_t* vo = final_pass ? col : vals[pass & 1];
        radix_hist<<<p.nblk, 256, 0, s>>>(src, p.n, shift, p.nblk, cnt);
        note_launch();
        cudaError_t e = launch_exclusive_scan(cnt, cnt, p.nscan, tmp, s, false);
        if (e != cudaSuccess) return e;
        radix_scatter<<<p.nblk, kRadixWarps * 32, smem, s>>>(src, p.n, shift, p.nblk, cnt, ko, vo);
        note_launch();
        src.keys = ko;
        src.vals = vo;
        last_keys = ko;
    }
    const int64_t threads = p.n + 1;
    csr_rowptr<<<unsigned((threads + 255) / 256), 256, 0, s>>>(last_keys, p.n, num_kv, row_ptr);
    note_launch();
    return cudaGetLastError();
}

}  // namespace smla
