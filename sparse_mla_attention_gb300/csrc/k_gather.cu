// k_gather.cu -- atomic-free dKV gather.
//
// The aiter page ("Sparse MLA training backward", Structure table, dKV gather)
// inverts the scatter so that each kv row gathers its own contributors from
// the [T, R, D] intermediate: dkv[j] = sum over CSR row j of interm[p].
// Rows are very unequal (a hot pool row can have thousands of contributors,
// a window row at most 128), so each row's list is cut into fixed segments of
// kGatherSeg entries. A warp sums one (segment, half of D) in CSR order into
// an fp32 partial; a second kernel adds a row's partials in segment order
// (and, in chunked mode, onto the fp32 accumulator of earlier chunks).
// Every addition has a fixed order, so dkv is bitwise reproducible.
#include "smla_internal.cuh"

namespace smla {

__global__ void seg_count(const int32_t* __restrict__ row_ptr, int num_kv,
                          int32_t* __restrict__ seg_cnt) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= num_kv) return;
    const int len = row_ptr[j + 1] - row_ptr[j];
    seg_cnt[j] = (len + kGatherSeg - 1) / kGatherSeg;
}

__global__ void seg_fill(const int32_t* __restrict__ seg_ptr, int num_kv,
                         int32_t* __restrict__ seg_row) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= num_kv) return;
    for (int s = seg_ptr[j]; s < seg_ptr[j + 1]; ++s) seg_row[s] = j;
}

// One warp per (segment, half of D); lane l owns 8 consecutive columns
// (one 16-byte load per contributor). The segment's contributor positions
// are loaded first, 8 per lane (one coalesced load each), and handed out by
// shuffles, so the interm loads do not wait on position loads; 8 interm loads
// per lane are in flight at a time. The additions run in CSR order.
__global__ void __launch_bounds__(256) seg_sum(const int32_t* __restrict__ row_ptr,
                                               const int32_t* __restrict__ col,
                                               const uint4* __restrict__ interm,
                                               const int32_t* __restrict__ seg_ptr,
                                               const int32_t* __restrict__ seg_row, int num_kv,
                                               float4* __restrict__ partial) {
    static_assert(kGatherSeg == 256, "a segment is 8 rounds of 32 positions");
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t sidx = gw >> 1;
    const int half = int(gw & 1);
    if (sidx >= seg_ptr[num_kv]) return;
    const int j = seg_row[sidx];
    const int local = int(sidx - seg_ptr[j]);
    const int e0 = row_ptr[j] + local * kGatherSeg;
    const int e1 = min(e0 + kGatherSeg, row_ptr[j + 1]);
    const int n = e1 - e0;
    int cl[8];                                    // cl[k] on lane l: position e0 + 32k + l
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int ee = e0 + 32 * k + lane;
        cl[k] = ee < e1 ? __ldg(col + ee) : 0;
    }
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    constexpr int kRowVec = kD * 2 / 16;          // 64 uint4 per interm row
    const int vcol = half * 32 + lane;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (32 * k >= n) break;
#pragma unroll
        for (int b = 0; b < 32; b += 8) {
            if (32 * k + b >= n) break;
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int pos = __shfl_sync(0xffffffffu, cl[k], b + u);
                v[u] = 32 * k + b + u < n ? __ldg(interm + int64_t(pos) * kRowVec + vcol)
                                          : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (32 * k + b + u >= n) break;
                const uint32_t* x = reinterpret_cast<const uint32_t*>(&v[u]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] += bf16_lo(x[q]);
                    acc[2 * q + 1] += bf16_hi(x[q]);
                }
            }
        }
    }
    float4* out = partial + sidx * (kD / 4) + half * 64 + lane * 2;
    out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// Thread per (kv row, 4 columns): adds the row's segment partials in order.
__global__ void __launch_bounds__(256) row_combine(const int32_t* __restrict__ seg_ptr,
                                                   const float4* __restrict__ partial, int num_kv,
                                                   float4* __restrict__ dkv_acc,
                                                   uint2* __restrict__ dkv_out, bool first,
                                                   bool last) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t j = i / (kD / 4);
    const int c = int(i % (kD / 4));
    if (j >= num_kv) return;
    float4 a = first ? make_float4(0.f, 0.f, 0.f, 0.f) : dkv_acc[j * (kD / 4) + c];
    for (int s = seg_ptr[j]; s < seg_ptr[j + 1]; ++s) {
        const float4 v = partial[int64_t(s) * (kD / 4) + c];
        a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
    }
    if (last)
        dkv_out[j * (kD / 4) + c] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
    else
        dkv_acc[j * (kD / 4) + c] = a;
}

cudaError_t launch_gather(const int32_t* row_ptr, const int32_t* col, const uint16_t* interm,
                          int num_kv, int64_t max_segs, int32_t* seg_cnt, int32_t* seg_ptr,
                          int32_t* seg_row, void* scan_tmp, float* partial, float* dkv_acc,
                          uint16_t* dkv_out, bool first_chunk, bool last_chunk, cudaStream_t s) {
    const unsigned gk = unsigned((num_kv + 255) / 256);
    seg_count<<<gk, 256, 0, s>>>(row_ptr, num_kv, seg_cnt);
    note_launch();
    cudaError_t e = launch_exclusive_scan(seg_cnt, seg_ptr, num_kv, scan_tmp, s, true);
    if (e != cudaSuccess) return e;
    seg_fill<<<gk, 256, 0, s>>>(seg_ptr, num_kv, seg_row);
    note_launch();
    if (max_segs > 0) {
        const int64_t warps = max_segs * 2;
        seg_sum<<<unsigned((warps * 32 + 255) / 256), 256, 0, s>>>(
            row_ptr, col, reinterpret_cast<const uint4*>(interm), seg_ptr, seg_row, num_kv,
            reinterpret_cast<float4*>(partial));
        note_launch();
    }
    const int64_t threads = int64_t(num_kv) * (kD / 4);
    row_combine<<<unsigned((threads + 255) / 256), 256, 0, s>>>(
        seg_ptr, reinterpret_cast<const float4*>(partial), num_kv,
        reinterpret_cast<float4*>(dkv_acc), reinterpret_cast<uint2*>(dkv_out), first_chunk,
        last_chunk);
    note_launch();
    return cudaGetLastError();
}

}  // namespace smla
