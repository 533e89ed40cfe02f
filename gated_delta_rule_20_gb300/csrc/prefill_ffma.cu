// prefill_ffma.cu -- chunk-parallel prefill of the gated delta-rule recurrence
// on FP32 FFMA.
//
// This is the fp32-compute path ("GDN CTE Kernel API Reference", Parameters /
// query: the query's dtype sets the compute dtype) and the path for head dims
// the tensor-core kernel does not cover.  Everything (operands, products, the
// triangular solve, the state) is fp32; bf16 inputs are widened on load.
//
// Chunk algebra (derived from the per-token recurrence; for a chunk of C tokens
// with start state S0, G_r = g_1 + ... + g_r inside the chunk, gamma_r = exp(G_r)):
//     A[r][j] = beta_r exp(G_r - G_j) k_r.k_j  (j < r)      T = (I + A)^-1
//     U = T diag(beta) V          W = T diag(beta gamma) K
//     Delta = U - W S0                                       (row r = delta_r)
//     O = scale (diag(gamma) Q S0 + P Delta),  P[r][j] = exp(G_r - G_j) q_r.k_j (j <= r)
//     S_end = gamma_C S0 + sum_j exp(G_C - G_j) k_j delta_j^T
// Every exponent that is evaluated is <= 0 (only j <= r pairs), so nothing
// overflows however strong the decay.  A ragged last chunk is padded with
// k = q = v = 0, g = 0, beta = 0 tokens, which leave the state unchanged.
//
// One CTA per (batch, value head), 256 threads, state resident in shared
// memory for the whole sequence; C = 32.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 32;
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float ld_f32(const T* p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void st_from_f32(T* p, float x);
template <>
__device__ __forceinline__ void st_from_f32<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_from_f32<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

struct Layout {
    int kpad;  // row stride of the K and Q tiles (Dk + 1: conflict-free column reads)
    int off_S, off_K, off_Q, off_V, off_W, off_U, off_A, off_T, off_P, off_small;
    int total_floats;
};

__host__ __device__ inline Layout make_layout(int Dk, int Dv) {
    Layout L;
    L.kpad = Dk + 1;
    int o = 0;
    L.off_S = o;  o += Dk * Dv;
    L.off_K = o;  o += kC * L.kpad;
    L.off_Q = o;  o += kC * L.kpad;
    L.off_V = o;  o += kC * Dv;
    L.off_W = o;  o += kC * Dk;
    L.off_U = o;  o += kC * Dv;
    L.off_A = o;  o += kC * (kC + 1);
    L.off_T = o;  o += kC * (kC + 1);
    L.off_P = o;  o += kC * (kC + 1);
    L.off_small = o; o += 4 * kC;
    L.total_floats = o;
    return L;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) gdn_prefill_ffma_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ g_log,
    const float* __restrict__ beta, float scale, float* __restrict__ state, T* __restrict__ out, int Hk, int Hv,
    int S, int Dk, int Dv, int zero_init) {
    extern __shared__ float smem[];
    const Layout L = make_layout(Dk, Dv);
    float* sS = smem + L.off_S;
    float* sK = smem + L.off_K;
    float* sQ = smem + L.off_Q;
    float* sV = smem + L.off_V;
    float* sW = smem + L.off_W;
    float* sU = smem + L.off_U;
    float* sA = smem + L.off_A;
    float* sT = smem + L.off_T;
    float* sP = smem + L.off_P;
    float* sG = smem + L.off_small;   // G_r
    float* sGam = sG + kC;            // gamma_r
    float* sBeta = sGam + kC;         // beta_r
    float* sEc = sBeta + kC;          // exp(G_C - G_r)
    constexpr int AP = kC + 1;

    const int bh = blockIdx.x;
    const int b = bh / Hv;
    const int h = bh - b * Hv;
    const int hk = h / (Hv / Hk);
    const int tid = threadIdx.x;

    const T* kb = k + (size_t)(b * Hk + hk) * S * Dk;
    const T* qb = q + (size_t)(b * Hk + hk) * S * Dk;
    const T* vb = v + (size_t)bh * S * Dv;
    const float* gb = g_log + (size_t)bh * S;
    const float* betab = beta + (size_t)bh * S;
    T* ob = out + (size_t)bh * S * Dv;
    float* Sg = state + (size_t)bh * Dk * Dv;

    for (int i = tid; i < Dk * Dv; i += kThreads) sS[i] = zero_init ? 0.f : Sg[i];

    for (int t0 = 0; t0 < S; t0 += kC) {
        const int n = min(kC, S - t0);
        __syncthreads();
        // ---- load the chunk (zero-padded past the end of the sequence)
        for (int i = tid; i < kC * Dk; i += kThreads) {
            const int r = i / Dk, d = i - r * Dk;
            const bool in = r < n;
            sK[r * L.kpad + d] = in ? ld_f32(kb + (size_t)(t0 + r) * Dk + d) : 0.f;
            sQ[r * L.kpad + d] = in ? ld_f32(qb + (size_t)(t0 + r) * Dk + d) : 0.f;
        }
        for (int i = tid; i < kC * Dv; i += kThreads) {
            const int r = i / Dv, c = i - r * Dv;
            sV[i] = (r < n) ? ld_f32(vb + (size_t)(t0 + r) * Dv + c) : 0.f;
        }
        if (tid < 32) {  // decay scan inside the chunk (kC == 32: one warp)
            const int r = tid;
            float gr = (r < n) ? gb[t0 + r] : 0.f;
            const float br = (r < n) ? betab[t0 + r] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float up = __shfl_up_sync(0xffffffffu, gr, o);
                if (r >= o) gr += up;
            }
            const float glast = __shfl_sync(0xffffffffu, gr, 31);
            sG[r] = gr;
            sGam[r] = expf(gr);
            sBeta[r] = br;
            sEc[r] = expf(glast - gr);
        }
        __syncthreads();

        // ---- A (strictly lower) and P (lower) from K K^T and Q K^T
        for (int i = tid; i < kC * kC; i += kThreads) {
            const int r = i / kC, j = i - r * kC;
            float a = 0.f, p = 0.f;
            if (j <= r) {
                float kk = 0.f, qk = 0.f;
                const float* kr = sK + r * L.kpad;
                const float* qr = sQ + r * L.kpad;
                const float* kj = sK + j * L.kpad;
                for (int d = 0; d < Dk; ++d) {
                    kk += kr[d] * kj[d];
                    qk += qr[d] * kj[d];
                }
                const float e = expf(sG[r] - sG[j]);
                p = e * qk;
                if (j < r) a = sBeta[r] * e * kk;
            }
            sA[r * AP + j] = a;
            sP[r * AP + j] = p;
        }
        __syncthreads();

        // ---- T = (I + A)^-1 by forward substitution, one column per thread
        if (tid < kC) {
            const int j = tid;
            float x[kC];
#pragma unroll
            for (int i = 0; i < kC; ++i) {
                float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < i; ++m) acc -= sA[i * AP + m] * x[m];
                x[i] = acc;
            }
#pragma unroll
            for (int i = 0; i < kC; ++i) sT[i * AP + j] = x[i];
        }
        __syncthreads();

        // ---- U = T diag(beta) V,  W = T diag(beta gamma) K
        for (int i = tid; i < kC * Dv; i += kThreads) {
            const int r = i / Dv, c = i - r * Dv;
            float acc = 0.f;
            for (int j = 0; j <= r; ++j) acc += sT[r * AP + j] * sBeta[j] * sV[j * Dv + c];
            sU[i] = acc;
        }
        for (int i = tid; i < kC * Dk; i += kThreads) {
            const int r = i / Dk, d = i - r * Dk;
            float acc = 0.f;
            for (int j = 0; j <= r; ++j) acc += sT[r * AP + j] * sBeta[j] * sGam[j] * sK[j * L.kpad + d];
            sW[i] = acc;
        }
        __syncthreads();

        // ---- Delta = U - W S0 (in place over U)
        for (int i = tid; i < kC * Dv; i += kThreads) {
            const int r = i / Dv, c = i - r * Dv;
            float acc = 0.f;
            for (int d = 0; d < Dk; ++d) acc += sW[r * Dk + d] * sS[d * Dv + c];
            sU[i] -= acc;
        }
        __syncthreads();

        // ---- O = scale (diag(gamma) Q S0 + P Delta)
        for (int i = tid; i < n * Dv; i += kThreads) {
            const int r = i / Dv, c = i - r * Dv;
            float qs = 0.f, pd = 0.f;
            for (int d = 0; d < Dk; ++d) qs += sQ[r * L.kpad + d] * sS[d * Dv + c];
            for (int j = 0; j <= r; ++j) pd += sP[r * AP + j] * sU[j * Dv + c];
            st_from_f32(ob + (size_t)(t0 + r) * Dv + c, scale * (sGam[r] * qs + pd));
        }
        __syncthreads();

        // ---- S = gamma_C S0 + sum_j exp(G_C - G_j) k_j delta_j^T
        const float gC = sGam[kC - 1];
        for (int i = tid; i < Dk * Dv; i += kThreads) {
            const int d = i / Dv, c = i - d * Dv;
            float acc = 0.f;
            for (int j = 0; j < kC; ++j) acc += sEc[j] * sK[j * L.kpad + d] * sU[j * Dv + c];
            sS[i] = gC * sS[i] + acc;
        }
    }
    __syncthreads();
    for (int i = tid; i < Dk * Dv; i += kThreads) Sg[i] = sS[i];
}

template <typename T>
cudaError_t launch_typed(const Problem& p, cudaStream_t stream) {
    const Layout L = make_layout(p.Dk, p.Dv);
    const size_t smem = (size_t)L.total_floats * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(gdn_prefill_ffma_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    gdn_prefill_ffma_kernel<T><<<p.B * p.Hv, kThreads, smem, stream>>>(
        static_cast<const T*>(p.q), static_cast<const T*>(p.k), static_cast<const T*>(p.v), p.g_log, p.beta,
        p.scale, p.state, static_cast<T*>(p.out), p.Hk, p.Hv, p.S, p.Dk, p.Dv, p.zero_init ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_ffma(const Problem& p, cudaStream_t stream) {
    return p.bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace gdn
