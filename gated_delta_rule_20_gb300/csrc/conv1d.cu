// conv1d.cu -- depthwise causal conv1d + SiLU in front of the recurrence, and
// its conv_state ("GDN Conv1D Kernel API Reference": gdn_conv1d_prefill and
// gdn_conv1d_decode; Parameters, Returns, Notes).
//
//   prefill: out[b, c, t] = silu(sum_{m=0}^{K-1} w[c, K-1-m] x[b, c, t-m]), x = 0 before t = 0;
//            conv_state[b, c, :] = the last K raw tokens (right-aligned behind zeros if T < K)
//   decode:  hs = (conv_state[b, c, 1:], x[b, c, 0]);  out = silu(sum_k w[c, k] hs[k]);
//            conv_state <- hs (in place)
//
// Both are bandwidth-bound streams: each activation is read once and written
// once.  The prefill's main path gives every lane 8 consecutive tokens of one
// channel (one 16-byte load and store of bf16) per step, several steps in flight,
// and takes the K - 1 <= 7 tokens before them from the neighbouring lane by a
// shuffle.  The decode step's common shape (bf16, K = 4) moves each window as one
// 8-byte word.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn.h"
#include "gdn_device.cuh"

namespace gdn {
namespace {

constexpr int kMaxTaps = 8;
constexpr int kThreadsPerBlock = 256;

__device__ __forceinline__ float silu(float z) { return silu_fast(z); }


__device__ __forceinline__ void unpack8(uint4 u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// bf16, T % 8 == 0, 16-byte aligned rows.  A warp covers kSeg = 32 * kUnroll
// consecutive 16-byte vectors (8 tokens each) of one (b, c) row: lane l takes the
// vectors seg_start + 32 u + l (coalesced), all loads issued before any math.
// The K - 1 <= 7 tokens before a lane's vector come from the lane before it (a
// shuffle); only lane 0 of the first group loads the vector before the segment.
constexpr int kUnroll = 4;
constexpr int kSeg = 32 * kUnroll;

__device__ __forceinline__ uint4 shfl_up4(uint4 v, int d) {
    return make_uint4(__shfl_up_sync(0xffffffffu, v.x, d), __shfl_up_sync(0xffffffffu, v.y, d),
                      __shfl_up_sync(0xffffffffu, v.z, d), __shfl_up_sync(0xffffffffu, v.w, d));
}
__device__ __forceinline__ uint4 shfl4(uint4 v, int src) {
    return make_uint4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                      __shfl_sync(0xffffffffu, v.z, src), __shfl_sync(0xffffffffu, v.w, src));
}

template <int K>  // taps, 1..8, fixed at compile time
__global__ void __launch_bounds__(kThreadsPerBlock) conv1d_prefill_vec8_kernel(
    const uint4* __restrict__ x, const float* __restrict__ w, uint4* __restrict__ out,
    __nv_bfloat16* __restrict__ state, int C, int nvec, int segs_per_row, long long n_warps) {
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (wid >= n_warps) return;  // whole warps leave together
    const int lane = threadIdx.x & 31;
    const long long row = wid / segs_per_row;  // b * C + c
    const int v0 = (int)(wid - row * segs_per_row) * kSeg;
    const int c = (int)(row % C);
    const uint4* xr = x + row * nvec;
    uint4 cur[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + 32 * u + lane;
        cur[u] = (v < nvec) ? xr[v] : make_uint4(0u, 0u, 0u, 0u);
    }
    const uint4 head = (lane == 0 && v0 > 0) ? xr[v0 - 1] : make_uint4(0u, 0u, 0u, 0u);
    float wb[K];  // wb[m] multiplies the token m steps back
#pragma unroll
    for (int m = 0; m < K; ++m) wb[m] = w[(long long)c * K + (K - 1 - m)];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        uint4 prev = shfl_up4(cur[u], 1);
        const uint4 last = (u > 0) ? shfl4(cur[u - 1], 31) : head;
        if (lane == 0) prev = last;
        float xx[16];  // tokens 8v - 8 .. 8v + 7
        unpack8(prev, xx);
        unpack8(cur[u], xx + 8);
        const int v = v0 + 32 * u + lane;
        if (v < nvec) {
            float y[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float z = 0.f;
#pragma unroll
                for (int m = 0; m < K; ++m) z = fmaf(wb[m], xx[8 + j - m], z);
                y[j] = silu(z);
            }
            out[row * nvec + v] =
                make_uint4(pack2(y[0], y[1]), pack2(y[2], y[3]), pack2(y[4], y[5]), pack2(y[6], y[7]));
            if (v == nvec - 1) {  // the row's last vector holds its last K raw tokens (T >= 8 >= K)
                const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(xr + v);
#pragma unroll
                for (int k = 0; k < K; ++k) state[row * K + k] = xv[8 - K + k];
            }
        }
    }
}

template <int K>
void launch_vec8(const void* mixed, const float* w, void* out, void* state, int C, int nvec, int segs,
                 long long n_warps, unsigned int blocks, cudaStream_t s) {
    conv1d_prefill_vec8_kernel<K><<<blocks, kThreadsPerBlock, 0, s>>>(
        static_cast<const uint4*>(mixed), w, static_cast<uint4*>(out), static_cast<__nv_bfloat16*>(state), C, nvec,
        segs, n_warps);
}

// Any dtype, T, alignment: one thread per (b, c, t).
template <typename T>
__global__ void __launch_bounds__(kThreadsPerBlock) conv1d_prefill_scalar_kernel(
    const T* __restrict__ x, const float* __restrict__ w, T* __restrict__ out, T* __restrict__ state, int C, int Tn,
    int K, long long total) {
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= total) return;
    const long long row = gid / Tn;
    const int t = (int)(gid - row * Tn);
    const int c = (int)(row % C);
    const T* xr = x + row * Tn;
    float z = 0.f;
    for (int m = 0; m < K && m <= t; ++m) z = fmaf(w[(long long)c * K + (K - 1 - m)], to_f32(xr[t - m]), z);
    out[gid] = from_f32<T>(silu(z));
    if (t >= Tn - K) state[row * K + (t - (Tn - K))] = xr[t];
    if (t == 0)
        for (int k = 0; k < K - Tn; ++k) state[row * K + k] = from_f32<T>(0.f);  // T < K: zeros in front
}

// One thread per (b, c) row: shift the window in place and take the K-tap dot product.
template <typename T>
__global__ void __launch_bounds__(kThreadsPerBlock) conv1d_decode_kernel(const T* __restrict__ x,
                                                                         const float* __restrict__ w,
                                                                         T* __restrict__ state, T* __restrict__ out,
                                                                         int C, int K, long long rows) {
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= rows) return;
    const int c = (int)(row % C);
    T* s = state + row * K;
    float z = 0.f;
    for (int k = 0; k < K; ++k) {  // reads s[k + 1] before s[k + 1] is rewritten
        const T hv = (k < K - 1) ? s[k + 1] : x[row];
        z = fmaf(w[(long long)c * K + k], to_f32(hv), z);
        s[k] = hv;
    }
    out[row] = from_f32<T>(silu(z));
}

// bf16, K == 4: the window is one 8-byte word (4 bf16) and the taps one float4.
__global__ void __launch_bounds__(kThreadsPerBlock) conv1d_decode_k4_kernel(const __nv_bfloat16* __restrict__ x,
                                                                            const float4* __restrict__ w,
                                                                            uint2* __restrict__ state,
                                                                            __nv_bfloat16* __restrict__ out, int C,
                                                                            long long rows) {
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= rows) return;
    const uint2 s = state[row];          // tokens s0 | s1 << 16, s2 | s3 << 16 (oldest first)
    const float4 wk = w[row % C];        // w[c, 0..3]
    const uint32_t xb = __bfloat16_as_ushort(x[row]);
    const float h0 = __uint_as_float(s.x & 0xffff0000u);  // s1
    const float h1 = __uint_as_float(s.y << 16);          // s2
    const float h2 = __uint_as_float(s.y & 0xffff0000u);  // s3
    const float h3 = __uint_as_float(xb << 16);           // the current token
    float z = fmaf(wk.x, h0, 0.f);
    z = fmaf(wk.y, h1, z);
    z = fmaf(wk.z, h2, z);
    z = fmaf(wk.w, h3, z);
    state[row] = make_uint2((s.x >> 16) | (s.y << 16), (s.y >> 16) | (xb << 16));
    out[row] = __float2bfloat16_rn(silu(z));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_conv(const void* x, const float* w, const void* state, const void* out, const gdn_conv_dims* d,
                      bool decode) {
    if (!d) return GDN_ERR_NULL;
    if (d->dtype != GDN_F32 && d->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (d->flags != 0) return GDN_ERR_UNSUPPORTED;
    if (d->B < 0 || d->C < 1 || d->T < 0 || d->K < 1) return GDN_ERR_DIMS;
    if (d->K > kMaxTaps) return GDN_ERR_UNSUPPORTED;
    if (decode && d->T != 1) return GDN_ERR_DIMS;
    if (d->B * d->C > INT32_MAX || d->T > INT32_MAX) return GDN_ERR_DIMS;
    if (d->B == 0) return GDN_OK;
    if (!w || !state) return GDN_ERR_NULL;
    if (d->T > 0 && (!x || !out)) return GDN_ERR_NULL;
    const size_t esz = d->dtype == GDN_BF16 ? 2 : 4;
    const uintptr_t mask = esz - 1;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(state)) & mask)
        return GDN_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(w) & 3u) return GDN_ERR_ALIGN;
    return GDN_OK;
}

unsigned int blocks_for(long long n) { return (unsigned int)((n + kThreadsPerBlock - 1) / kThreadsPerBlock); }

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_conv1d_prefill(const void* mixed, const float* conv_weight, void* out, void* conv_state_out,
                              const gdn_conv_dims* dims, gdn_stream_t stream) {
    const gdn_status st = check_conv(mixed, conv_weight, conv_state_out, out, dims, false);
    if (st != GDN_OK || dims->B == 0) return st;
    const long long rows = dims->B * dims->C;
    const int C = (int)dims->C, T = (int)dims->T, K = (int)dims->K;
    const bool bf16 = dims->dtype == GDN_BF16;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {  // no tokens: the last K raw tokens are all padding
        const size_t bytes = (size_t)rows * K * (bf16 ? 2 : 4);
        return cudaMemsetAsync(conv_state_out, 0, bytes, s) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (bf16 && T % 8 == 0 && aligned16(mixed) && aligned16(out)) {
        const int nvec = T / 8;
        const int segs = (nvec + kSeg - 1) / kSeg;
        const long long n_warps = rows * segs;
        const unsigned int blocks = blocks_for(n_warps * 32);
        switch (K) {
            case 1: launch_vec8<1>(mixed, conv_weight, out, conv_state_out, C, nvec, segs, n_warps, blocks, s); break;
            case 2: launch_vec8<2>(mixed, conv_weight, out, conv_state_out, C, nvec, segs, n_warps, blocks, s); break;
            case 3: launch_vec8<3>(mixed, conv_weight, out, conv_state_out, C, nvec, segs, n_warps, blocks, s); break;
            case 4: launch_vec8<4>(mixed, conv_weight, out, conv_state_out, C, nvec, segs, n_warps, blocks, s); break;
            case 5: launch_vec8<5>(mixed, conv_weight, out, conv_state_out, C, nvec, segs, n_warps, blocks, s); break;
            case 6: launch_vec8<6>(mixed, conv_weight, out, conv_state_out, C, nvec, segs, n_warps, blocks, s); break;
            case 7: launch_vec8<7>(mixed, conv_weight, out, conv_state_out, C, nvec, segs, n_warps, blocks, s); break;
            default: launch_vec8<8>(mixed, conv_weight, out, conv_state_out, C, nvec, segs, n_warps, blocks, s); break;
        }
    } else if (bf16) {
        const long long total = rows * T;
        conv1d_prefill_scalar_kernel<__nv_bfloat16><<<blocks_for(total), kThreadsPerBlock, 0, s>>>(
            static_cast<const __nv_bfloat16*>(mixed), conv_weight, static_cast<__nv_bfloat16*>(out),
            static_cast<__nv_bfloat16*>(conv_state_out), C, T, K, total);
    } else {
        const long long total = rows * T;
        conv1d_prefill_scalar_kernel<float><<<blocks_for(total), kThreadsPerBlock, 0, s>>>(
            static_cast<const float*>(mixed), conv_weight, static_cast<float*>(out),
            static_cast<float*>(conv_state_out), C, T, K, total);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_conv1d_decode(const void* x, const float* conv_weight, void* conv_state_inout, void* out,
                             const gdn_conv_dims* dims, gdn_stream_t stream) {
    const gdn_status st = check_conv(x, conv_weight, conv_state_inout, out, dims, true);
    if (st != GDN_OK || dims->B == 0) return st;
    const long long rows = dims->B * dims->C;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dims->dtype == GDN_BF16 && dims->K == 4 && aligned16(conv_weight) &&
        (reinterpret_cast<uintptr_t>(conv_state_inout) & 7u) == 0) {
        conv1d_decode_k4_kernel<<<blocks_for(rows), kThreadsPerBlock, 0, s>>>(
            static_cast<const __nv_bfloat16*>(x), reinterpret_cast<const float4*>(conv_weight),
            static_cast<uint2*>(conv_state_inout), static_cast<__nv_bfloat16*>(out), (int)dims->C, rows);
    } else if (dims->dtype == GDN_BF16) {
        conv1d_decode_kernel<__nv_bfloat16><<<blocks_for(rows), kThreadsPerBlock, 0, s>>>(
            static_cast<const __nv_bfloat16*>(x), conv_weight, static_cast<__nv_bfloat16*>(conv_state_inout),
            static_cast<__nv_bfloat16*>(out), (int)dims->C, (int)dims->K, rows);
    } else {
        conv1d_decode_kernel<float><<<blocks_for(rows), kThreadsPerBlock, 0, s>>>(
            static_cast<const float*>(x), conv_weight, static_cast<float*>(conv_state_inout),
            static_cast<float*>(out), (int)dims->C, (int)dims->K, rows);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
