// rmsnorm_gated.cu -- the RMSNormGated output epilogue as a row pass, and the
// gated prefill built on it ("GDN Block TKG Kernel API Reference": Returns,
// "RMSNormGated decode output", and the norm_weight parameter, "RMSNormGated
// weight"; applied here to every token of a prefill, whose un-normalised output
// the "GDN CTE Kernel API Reference" Returns section describes).
//
//     y[r, :] = x[r, :] / sqrt(mean(x[r, :]^2) + eps) * norm_weight * silu(z[r, :])
//
// over rows of D elements (a value head's Dv outputs of one token).  The pass
// reads x and z once and writes y once (in place is allowed), so it is bound by
// HBM.  D = 128 with 16-byte aligned rows: 16 bytes per lane per row (a half
// warp per bf16 row, a warp per fp32 row), and each warp issues the loads of
// kRowIters row groups before it computes any, so that enough bytes are in
// flight.  Other D take a scalar loop, one warp per row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn_internal.h"
#include "gdn_device.cuh"

namespace gdn {
namespace {

constexpr int kRowsPerBlock = 8;  // scalar kernel: one warp per row, 256 threads
constexpr int kRowIters = 4;      // D = 128 kernel: row groups per warp
constexpr float kEps = GDN_RMSNORM_EPS;

__device__ __forceinline__ float silu(float z) { return silu_fast(z); }


// D = 128, 16-byte aligned: a row is kLanes lanes x 8 (bf16) or 4 (fp32) elements; a warp
// holds 32 / kLanes rows at a time and kRowIters such groups.
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_gated_d128_kernel(const T* x, const T* z, const float* __restrict__ w,
                                                                 T* y, long long rows) {
    constexpr int kPer = 16 / (int)sizeof(T);  // elements per lane
    constexpr int kLanes = 128 / kPer;         // lanes per row: 16 (bf16) or 32 (fp32)
    constexpr int kRowsPerWarp = 32 / kLanes;
    const int lane = threadIdx.x & 31, sub = lane % kLanes;
    const long long warp = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const long long r0 = warp * (kRowsPerWarp * kRowIters) + lane / kLanes;
    uint4 xv[kRowIters], zv[kRowIters];
#pragma unroll
    for (int it = 0; it < kRowIters; ++it) {
        const long long r = r0 + (long long)it * kRowsPerWarp;
        if (r < rows) {
            xv[it] = *reinterpret_cast<const uint4*>(x + r * 128 + kPer * sub);
            zv[it] = *reinterpret_cast<const uint4*>(z + r * 128 + kPer * sub);
        }
    }
    float wv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; j += 4) {
        const float4 t = *reinterpret_cast<const float4*>(w + kPer * sub + j);
        wv[j] = t.x;
        wv[j + 1] = t.y;
        wv[j + 2] = t.z;
        wv[j + 3] = t.w;
    }
#pragma unroll
    for (int it = 0; it < kRowIters; ++it) {
        const long long r = r0 + (long long)it * kRowsPerWarp;
        float a[kPer], b[kPer];
        const T* xa = reinterpret_cast<const T*>(&xv[it]);
        const T* za = reinterpret_cast<const T*>(&zv[it]);
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            a[j] = to_f32(xa[j]);
            b[j] = to_f32(za[j]);
            ss += a[j] * a[j];
        }
#pragma unroll
        for (int o = kLanes / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);  // within the row
        const float rinv = rsqrtf(ss / 128.f + kEps);
        if (r < rows) {
            uint4 ov;
            T* oa = reinterpret_cast<T*>(&ov);
#pragma unroll
            for (int j = 0; j < kPer; ++j) oa[j] = from_f32<T>(a[j] * rinv * wv[j] * silu(b[j]));
            *reinterpret_cast<uint4*>(y + r * 128 + kPer * sub) = ov;
        }
    }
}

// any D: lane l owns elements l, l + 32, ...
template <typename T>
__global__ void __launch_bounds__(32 * kRowsPerBlock) rmsnorm_gated_kernel(const T* x, const T* z,
                                                                           const float* __restrict__ w, T* y,
                                                                           long long rows, int D) {
    const long long r = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int lane = threadIdx.x & 31;
    float ss = 0.f;
    for (int i = lane; i < D; i += 32) {
        const float v = to_f32(x[r * D + i]);
        ss += v * v;
    }
    const float rinv = rsqrtf(warp_sum(ss) / (float)D + kEps);
    for (int i = lane; i < D; i += 32)
        y[r * D + i] = from_f32<T>(to_f32(x[r * D + i]) * rinv * w[i] * silu(to_f32(z[r * D + i])));
}

gdn_status check_norm(const void* x, const void* z, const float* w, const void* y, long long rows, long long D,
                      int32_t dtype) {
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (rows < 0 || D < 1 || D > 4096) return GDN_ERR_DIMS;
    if (rows == 0) return GDN_OK;
    if (!x || !z || !w || !y) return GDN_ERR_NULL;
    const uintptr_t esz = dtype == GDN_BF16 ? 2 : 4;
    if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(y)) &
         (esz - 1)) ||
        (reinterpret_cast<uintptr_t>(w) & 3u))
        return GDN_ERR_ALIGN;
    return GDN_OK;
}

template <typename T>
cudaError_t launch_norm(const void* x, const void* z, const float* w, void* y, long long rows, int D,
                        cudaStream_t s) {
    const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const bool vec = D == 128 && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(z) |
                                   reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(w)) & 15u) == 0;
    if (vec) {
        const long long rows_per_block = 8LL * (32 / (128 / (16 / (long long)sizeof(T)))) * kRowIters;
        rmsnorm_gated_d128_kernel<T><<<(unsigned)((rows + rows_per_block - 1) / rows_per_block), 256, 0, s>>>(
            static_cast<const T*>(x), static_cast<const T*>(z), w, static_cast<T*>(y), rows);
    } else
        rmsnorm_gated_kernel<T><<<(unsigned)blocks, 32 * kRowsPerBlock, 0, s>>>(
            static_cast<const T*>(x), static_cast<const T*>(z), w, static_cast<T*>(y), rows, D);
    return cudaGetLastError();
}

cudaError_t run_norm(const void* x, const void* z, const float* w, void* y, long long rows, int D, int32_t dtype,
                     cudaStream_t s) {
    return dtype == GDN_BF16 ? launch_norm<__nv_bfloat16>(x, z, w, y, rows, D, s)
                             : launch_norm<float>(x, z, w, y, rows, D, s);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_rmsnorm_gated(const void* x, const void* z, const float* norm_weight, void* out,
                                        int64_t rows, int64_t D, int32_t dtype, gdn_stream_t stream) {
    const gdn_status st = check_norm(x, z, norm_weight, out, rows, D, dtype);
    if (st != GDN_OK || rows == 0) return st;
    if ((rows + kRowsPerBlock - 1) / kRowsPerBlock > INT32_MAX) return GDN_ERR_DIMS;
    return run_norm(x, z, norm_weight, out, rows, (int)D, dtype, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_prefill_gated(const void* q, const void* k, const void* v, const float* g_log,
                                        const float* beta, const void* z, const float* norm_weight, float scale,
                                        float* state_inout, void* out, const gdn_dims* dims, gdn_stream_t stream) {
    if (!dims) return GDN_ERR_NULL;
    const long long rows = dims->B * dims->Hv * dims->S;
    // every check of both steps runs before the first launch
    gdn_status st = prefill_checked(q, k, v, g_log, beta, state_inout, out, dims);
    if (st != GDN_OK) return st;
    if (rows > 0) {
        st = check_norm(out, z, norm_weight, out, rows, dims->Dv, dims->dtype);
        if (st != GDN_OK) return st;
        if ((rows + kRowsPerBlock - 1) / kRowsPerBlock > INT32_MAX) return GDN_ERR_DIMS;
    }
    st = gdn_prefill(q, k, v, g_log, beta, scale, state_inout, out, dims, stream);
    if (st != GDN_OK || rows == 0) return st;
    return run_norm(out, z, norm_weight, out, rows, (int)dims->Dv, dims->dtype,
                    reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}
