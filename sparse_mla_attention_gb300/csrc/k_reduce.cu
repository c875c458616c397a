// k_reduce.cu -- bandwidth-bound phases of the sparse MLA backward:
//   * delta = rowsum(O * dO)            (the page's "delta" phase)
//   * d_sink = -sum_t exp(sink - lse) * delta   (the page's "d_sink" phase)
//   * a generic device-wide exclusive scan of int32 counts.
// Source: aiter "[WIP][TRITON][GLUON][GFX950][DSV4] Sparse MLA training
// backward", Structure table (delta streams bf16 and accumulates in fp32;
// d_sink is a reduction over tokens).
#include "smla_internal.cuh"

namespace smla {

// ------------------------------------------------------------------- delta
// One warp per (t, h) row of 512 bf16: each lane loads 2 x 16 B of O and of
// dO (128-bit vector loads), forms 16 products in fp32 and the warp reduces
// them with shuffles. Rows are walked grid-stride, two per warp iteration so
// that four 16-byte loads per lane are in flight.
__global__ void __launch_bounds__(256) delta_kernel(const uint4* __restrict__ o,
                                                    const uint4* __restrict__ dO,
                                                    float* __restrict__ delta, int64_t rows) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    constexpr int kVec = kD * 2 / 16;  // 64 uint4 per row
    for (int64_t r0 = warp * 2; r0 < rows; r0 += nwarps * 2) {
        float acc[2] = {0.f, 0.f};
        uint4 a[2][2], b[2][2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int64_t r = r0 + k;
            if (r < rows) {
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    a[k][v] = __ldcs(o + r * kVec + v * 32 + lane);
                    b[k][v] = __ldcs(dO + r * kVec + v * 32 + lane);
                }
            } else {
#pragma unroll
                for (int v = 0; v < 2; ++v) a[k][v] = b[k][v] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const uint32_t* x = reinterpret_cast<const uint32_t*>(&a[k][v]);
                const uint32_t* y = reinterpret_cast<const uint32_t*>(&b[k][v]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[k] = fmaf(bf16_lo(x[e]), bf16_lo(y[e]), acc[k]);
                    acc[k] = fmaf(bf16_hi(x[e]), bf16_hi(y[e]), acc[k]);
                }
            }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
            if (lane == 0 && r0 + k < rows) delta[r0 + k] = acc[k];
        }
    }
}

cudaError_t launch_delta(const uint16_t* o, const uint16_t* dO, float* delta,
                         int64_t rows, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (rows + 15) / 16;      // blocks of 8 warps x 2 rows
    const int grid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    delta_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(o),
                                      reinterpret_cast<const uint4*>(dO), delta, rows);
    note_launch();
    return cudaGetLastError();
}

// ------------------------------------------------------------------ d_sink
// One block of 8 warps per head. Thread i sums tokens i, i+256, ... in
// ascending order; each warp then combines its 32 partials with a butterfly
// of shuffles, and warp 0 combines the 8 warp sums the same way. Every
// addition has a fixed place in that tree, so the result is bitwise
// reproducible.
// Term: the sink's softmax weight exp(sink_h - lse) times (0 - delta), the
// sink having no value row.
__device__ __forceinline__ float warp_sum_fixed(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__global__ void __launch_bounds__(256) dsink_kernel(const float* __restrict__ delta,
                                                    const float* __restrict__ lse,
                                                    const float* __restrict__ sink,
                                                    float* __restrict__ d_sink, int T, int H) {
    __shared__ float warp_part[8];
    const int h = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float sh = sink[h];
    float acc = 0.f;
    for (int t = threadIdx.x; t < T; t += 256) {
        const float l = lse[int64_t(t) * H + h];
        acc -= expf(sh - l) * delta[int64_t(t) * H + h];
    }
    acc = warp_sum_fixed(acc);
    if (lane == 0) warp_part[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        float v = lane < 8 ? warp_part[lane] : 0.f;
        v = warp_sum_fixed(v);
        if (lane == 0) d_sink[h] = v;
    }
}

cudaError_t launch_dsink(const float* delta, const float* lse, const float* sink,
                         float* d_sink, int T, int H, cudaStream_t s) {
    dsink_kernel<<<H, 256, 0, s>>>(delta, lse, sink, d_sink, T, H);
    note_launch();
    return cudaGetLastError();
}

// --------------------------------------------------------- ordered partials
// The combine step of a token-sharded backward: every element is the sum of
// the ranks' partials taken in rank order (a fixed order, so every rank that
// runs this on the same gathered partials gets the same bits). One thread per
// 4 consecutive elements, grid-stride.
__global__ void __launch_bounds__(256) reduce_partials_kernel(const float4* __restrict__ parts,
                                                              int n_parts, int64_t n4,
                                                              uint2* __restrict__ out_bf16,
                                                              float4* __restrict__ out_f32) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        float4 a = parts[i];
        for (int r = 1; r < n_parts; ++r) {
            const float4 v = parts[int64_t(r) * n4 + i];
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
        if (out_f32) out_f32[i] = a;
        if (out_bf16) out_bf16[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
    }
}

cudaError_t launch_reduce_partials(const float* partials, int n_parts, int64_t n,
                                   uint16_t* out_bf16, float* out_f32, cudaStream_t s) {
    const int64_t n4 = n / 4;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (n4 + 255) / 256;
    const int grid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    reduce_partials_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(
        reinterpret_cast<const float4*>(partials), n_parts, n4, reinterpret_cast<uint2*>(out_bf16),
        reinterpret_cast<float4*>(out_f32));
    note_launch();
    return cudaGetLastError();
}

// ------------------------------------------------------------ exclusive scan
// Reduce-then-scan over tiles of 2048 int32 (256 threads x 8): tile sums,
// then one block scans the tile sums (looping when there are more than
// 2048 tiles), then each tile scans itself and adds its tile offset.
constexpr int kScanTile = 2048;

size_t scan_tmp_bytes(int64_t n) {
    const int64_t tiles = (n + kScanTile - 1) / kScanTile;
    return align_up(size_t(tiles + 1) * sizeof(int32_t), 256);
}

__device__ __forceinline__ int block_exclusive_scan_256(int v, int* sh, int* total) {
    // inclusive warp scan
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < 8 ? sh[lane] : 0;
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        if (lane < 8) sh[lane] = w;
    }
    __syncthreads();
    const int before = (warp > 0 ? sh[warp - 1] : 0) + x - v;
    if (total) *total = sh[7];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(256) scan_tile_sums(const int32_t* __restrict__ in,
                                                      int32_t* __restrict__ sums, int64_t n) {
    __shared__ int sh[8];
    const int64_t base = int64_t(blockIdx.x) * kScanTile + threadIdx.x * 8;
    int v = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (base + k < n) v += in[base + k];
    int total;
    block_exclusive_scan_256(v, sh, &total);
    if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

__global__ void __launch_bounds__(256) scan_sums(int32_t* __restrict__ sums, int64_t tiles) {
    __shared__ int sh[8];
    int carry = 0;
    for (int64_t b0 = 0; b0 < tiles; b0 += kScanTile) {
        int v[8];
        int local = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t i = b0 + threadIdx.x * 8 + k;
            v[k] = i < tiles ? sums[i] : 0;
            local += v[k];
        }
        int total;
        int run = carry + block_exclusive_scan_256(local, sh, &total);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t i = b0 + threadIdx.x * 8 + k;
            if (i < tiles) sums[i] = run;
            run += v[k];
        }
        carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) sums[tiles] = carry;
}

__global__ void __launch_bounds__(256) scan_apply(const int32_t* in, int32_t* out,
                                                  const int32_t* __restrict__ sums, int64_t n,
                                                  int64_t tiles, bool write_total) {
    __shared__ int sh[8];
    if (write_total && blockIdx.x == 0 && threadIdx.x == 0) out[n] = sums[tiles];
    const int64_t base = int64_t(blockIdx.x) * kScanTile + threadIdx.x * 8;
    int v[8];
    int local = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[k] = base + k < n ? in[base + k] : 0;
        local += v[k];
    }
    int run = sums[blockIdx.x] + block_exclusive_scan_256(local, sh, nullptr);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (base + k < n) out[base + k] = run;
        run += v[k];
    }
}

// out[i] = sum of in[0..i) for i in [0, n); with write_total, also
// out[n] = sum of all n values (the caller sized `out` for n + 1 entries).
// `in` and `out` may be the same buffer.
cudaError_t launch_exclusive_scan(const int32_t* in, int32_t* out, int64_t n, void* tmp,
                                  cudaStream_t s, bool write_total) {
    if (n <= 0) {
        if (write_total) return cudaMemsetAsync(out, 0, sizeof(int32_t), s);
        return cudaSuccess;
    }
    const int64_t tiles = (n + kScanTile - 1) / kScanTile;
    int32_t* sums = static_cast<int32_t*>(tmp);
    scan_tile_sums<<<unsigned(tiles), 256, 0, s>>>(in, sums, n);
    note_launch();
    scan_sums<<<1, 256, 0, s>>>(sums, tiles);
    note_launch();
    scan_apply<<<unsigned(tiles), 256, 0, s>>>(in, out, sums, n, tiles, write_total);
    note_launch();
    return cudaGetLastError();
}

}  // namespace smla
