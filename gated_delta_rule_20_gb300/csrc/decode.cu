// decode.cu -- single-token step of the gated delta-rule recurrence.
//
// The recurrence at S = 1 ("GDN Block TKG Kernel API Reference": the
// single-token recurrence inside gdn_tkg, recurrent_state
// [B, num_v_heads, head_k_dim, head_v_dim] fp32):
//
//     a  = exp(g);  p_k = S^T k;  p_q = S^T q
//     d  = beta (v - a p_k)
//     o  = scale S'^T q = scale (a p_q + d (k . q))
//     S' = a S + k d^T                  (written back in place)
//
// The state dominates the traffic (64 KiB per head at Dk = Dv = 128), so the
// kernel is built around one coalesced pass: every fp32 state element is loaded
// once with a 128-bit load into registers, reduced, updated and stored once.
//
// Dk = Dv = 128 runs gdn_decode_stream_kernel (below): persistent CTAs that
// bulk-copy the next head's state into shared memory while they compute the
// current one.  Other head dims run gdn_decode_kernel.  Grid: (B * Hv,
// ceil(Dv / 64)).  A CTA owns one 64-column slice of one head's state (columns
// evolve independently: column c of S' depends only on column c of S).  128
// threads = 16 column groups of 4 floats x 8 row groups; thread (rg, cg) holds
// rows rg, rg + 8, ... of its 4 columns.  A warp therefore reads two full
// 256-byte row segments per load instruction.  Four CTAs share an SM (128
// registers per thread), so that more state loads are in flight.
#include <cuda_bf16.h>

#include <mutex>

#include "gdn_internal.h"
#include "gdn_device.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

constexpr int kCols = 64;         // state columns per CTA
constexpr int kThreads = 128;     // 16 column groups x 8 row groups
constexpr int kRowGroups = 8;
constexpr int kMaxRowsPerThread = 128 / kRowGroups;

template <typename T, bool kVec>
__global__ void __launch_bounds__(kThreads, 4) gdn_decode_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                              const T* __restrict__ v,
                                                              const float* __restrict__ g_log,
                                                              const float* __restrict__ beta, float scale,
                                                              float* __restrict__ state, T* __restrict__ out,
                                                              int Hk, int Hv, int Dk, int Dv, int zero_init) {
    __shared__ float s_k[128];
    __shared__ float s_q[128];
    __shared__ float s_red[2][kRowGroups][kCols];
    __shared__ float s_d[kCols];
    __shared__ float s_kq;

    const int bh = blockIdx.x;            // b * Hv + h
    const int b = bh / Hv;
    const int h = bh - b * Hv;
    const int hk = h / (Hv / Hk);         // blocked GQA mapping
    const int c_base = blockIdx.y * kCols;
    const int tid = threadIdx.x;
    const int cg = tid & 15;              // column group: 4 columns
    const int rg = tid >> 4;              // row group
    const int c0 = c_base + cg * 4;

    const T* kp = k + (size_t)(b * Hk + hk) * Dk;
    const T* qp = q + (size_t)(b * Hk + hk) * Dk;
    float* Sp = state + (size_t)bh * Dk * Dv;

    // Issue the state loads first: they are the bulk of the traffic.
    float4 S[kMaxRowsPerThread];
#pragma unroll
    for (int i = 0; i < kMaxRowsPerThread; ++i) {
        const int r = rg + i * kRowGroups;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!zero_init && r < Dk) {
            if (kVec) {
                if (c0 < Dv) x = __ldcs(reinterpret_cast<const float4*>(Sp + (size_t)r * Dv + c0));
            } else {
                const float* row = Sp + (size_t)r * Dv;
                if (c0 + 0 < Dv) x.x = row[c0 + 0];
                if (c0 + 1 < Dv) x.y = row[c0 + 1];
                if (c0 + 2 < Dv) x.z = row[c0 + 2];
                if (c0 + 3 < Dv) x.w = row[c0 + 3];
            }
        }
        S[i] = x;
    }

    // the value row is fetched now too, so that its load does not wait behind a barrier
    const int cv = c_base + (tid & (kCols - 1));
    const float vc = (tid < kCols && cv < Dv) ? to_f32(v[(size_t)bh * Dv + cv]) : 0.f;
    if (tid < Dk) {
        s_k[tid] = to_f32(kp[tid]);
        s_q[tid] = to_f32(qp[tid]);
    }
    const float a = expf(g_log[bh]);
    const float bt = beta[bh];
    __syncthreads();
    if (tid < 32) {  // k . q
        float acc = 0.f;
        for (int i = tid; i < Dk; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (tid == 0) s_kq = acc;
    }

    // Partial S^T k and S^T q over this thread's rows.
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kMaxRowsPerThread; ++i) {
        const int r = rg + i * kRowGroups;
        if (r < Dk) {
            const float kr = s_k[r], qr = s_q[r];
            pk[0] += S[i].x * kr; pk[1] += S[i].y * kr; pk[2] += S[i].z * kr; pk[3] += S[i].w * kr;
            pq[0] += S[i].x * qr; pq[1] += S[i].y * qr; pq[2] += S[i].z * qr; pq[3] += S[i].w * qr;
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s_red[0][rg][cg * 4 + j] = pk[j];
        s_red[1][rg][cg * 4 + j] = pq[j];
    }
    __syncthreads();
    if (tid < kCols) {
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int g = 0; g < kRowGroups; ++g) {
            sk += s_red[0][g][tid];
            sq += s_red[1][g][tid];
        }
        const int c = c_base + tid;
        const float d = bt * (vc - a * sk);
        s_d[tid] = d;
        if (c < Dv) out[(size_t)bh * Dv + c] = from_f32<T>(scale * (a * sq + d * s_kq));
    }
    __syncthreads();

    const float d0 = s_d[cg * 4 + 0], d1 = s_d[cg * 4 + 1], d2 = s_d[cg * 4 + 2], d3 = s_d[cg * 4 + 3];
#pragma unroll
    for (int i = 0; i < kMaxRowsPerThread; ++i) {
        const int r = rg + i * kRowGroups;
        if (r < Dk) {
            const float kr = s_k[r];
            float4 x;
            x.x = a * S[i].x + kr * d0;
            x.y = a * S[i].y + kr * d1;
            x.z = a * S[i].z + kr * d2;
            x.w = a * S[i].w + kr * d3;
            if (kVec) {
                if (c0 < Dv) __stcs(reinterpret_cast<float4*>(Sp + (size_t)r * Dv + c0), x);
            } else {
                float* row = Sp + (size_t)r * Dv;
                if (c0 + 0 < Dv) row[c0 + 0] = x.x;
                if (c0 + 1 < Dv) row[c0 + 1] = x.y;
                if (c0 + 2 < Dv) row[c0 + 2] = x.z;
                if (c0 + 3 < Dv) row[c0 + 3] = x.w;
            }
        }
    }
}

// Dk = Dv = 128: persistent CTAs, two per SM, walk the heads blockIdx.x, blockIdx.x +
// gridDim.x, ...  A head's state (64 KB) reaches shared memory in one bulk copy and its q,
// k, v rows in 16-byte asynchronous copies, both issued as soon as the previous head has
// been read out of shared memory, so that the memory system holds the next head's bytes
// while the CTA computes.  256 threads = 32 column groups of 4 x 8 row groups; each state
// element is still read once and written once.
constexpr int kSD = 128;
constexpr int kSThreads = 256;
constexpr int kSColGroups = 32;
constexpr uint32_t kSStateBytes = kSD * kSD * 4;

struct DecodeStreamSmem {
    float state[kSD * kSD];
    alignas(16) uint8_t in[3 * kSD * 4];  // q, k, v rows in the compute type
    uint64_t full;
    int abort;
};

template <typename T>
__global__ void __launch_bounds__(kSThreads, 2) gdn_decode_stream_kernel(Problem p, int32_t* status) {
    extern __shared__ __align__(128) uint8_t decode_raw[];
    DecodeStreamSmem& sm = *reinterpret_cast<DecodeStreamSmem*>(decode_raw);
    __shared__ float s_k[kSD], s_q[kSD];
    __shared__ float s_red[2][kRowGroups][kSD];
    __shared__ float s_d[kSD];
    __shared__ float s_kq;
    const int tid = threadIdx.x;
    const int cg = tid & (kSColGroups - 1), rg = tid >> 5, c0 = cg * 4;
    const int heads = p.B * p.Hv;
    const int n_local = (heads - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    auto head_of = [&](int l) { return (int)blockIdx.x + l * (int)gridDim.x; };
    auto load_state = [&](int bh) {
        ptx::mbar_arrive_expect_tx(&sm.full, kSStateBytes);
        ptx::bulk_load_evict_first(sm.state, p.state + (size_t)bh * kSD * kSD, kSStateBytes, &sm.full);
    };
    // q, k (key head h / (Hv / Hk)) and v rows of head bh: 3 x 128 elements
    auto load_inputs = [&](int bh) {
        const int b = bh / p.Hv, h = bh - b * p.Hv, hk = h / (p.Hv / p.Hk);
        const uint8_t* qr = static_cast<const uint8_t*>(p.q) + (size_t)(b * p.Hk + hk) * kSD * sizeof(T);
        const uint8_t* kr = static_cast<const uint8_t*>(p.k) + (size_t)(b * p.Hk + hk) * kSD * sizeof(T);
        const uint8_t* vr = static_cast<const uint8_t*>(p.v) + (size_t)bh * kSD * sizeof(T);
        constexpr int kChunks = kSD * (int)sizeof(T) / 16;  // per row
        for (int i = tid; i < 3 * kChunks; i += kSThreads) {
            const int r = i / kChunks, c = i % kChunks;
            const uint8_t* src = r == 0 ? qr : r == 1 ? kr : vr;
            ptx::cp_async_16(sm.in + r * kSD * sizeof(T) + 16 * c, src + 16 * c);
        }
        ptx::cp_async_commit();
    };
    if (tid == 0) {
        ptx::mbar_init(&sm.full, 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0 && !p.zero_init) load_state(head_of(0));
    load_inputs(head_of(0));
    float g_n = p.g_log[head_of(0)], b_n = p.beta[head_of(0)];

    for (int l = 0; l < n_local; ++l) {
        const int bh = head_of(l);
        const float a = expf(g_n), bt = b_n;
        if (!p.zero_init) (void)ptx::mbar_wait_or_abort(&sm.full, l & 1, &sm.abort);
        ptx::cp_async_wait_all();
        __syncthreads();  // every thread's copies have landed; the previous head is done with the scratch
        float4 S[kMaxRowsPerThread];
#pragma unroll
        for (int i = 0; i < kMaxRowsPerThread; ++i)
            S[i] = p.zero_init ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : *reinterpret_cast<const float4*>(&sm.state[(rg + i * kRowGroups) * kSD + c0]);
        if (tid < kSD) {
            const T* in = reinterpret_cast<const T*>(sm.in);
            s_q[tid] = to_f32(in[tid]);
            s_k[tid] = to_f32(in[kSD + tid]);
            s_d[tid] = to_f32(in[2 * kSD + tid]);  // v, until d replaces it
        }
        __syncthreads();  // the state and the inputs of head l have been read out of shared memory
        if (l + 1 < n_local) {
            const int nb = head_of(l + 1);
            if (tid == 0 && !p.zero_init) load_state(nb);
            load_inputs(nb);
            g_n = p.g_log[nb];
            b_n = p.beta[nb];
        }
        if (tid < 32) {  // k . q
            float acc = 0.f;
            for (int i = tid; i < kSD; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (tid == 0) s_kq = acc;
        }
        float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kMaxRowsPerThread; ++i) {
            const int r = rg + i * kRowGroups;
            const float kr = s_k[r], qr = s_q[r];
            pk[0] += S[i].x * kr; pk[1] += S[i].y * kr; pk[2] += S[i].z * kr; pk[3] += S[i].w * kr;
            pq[0] += S[i].x * qr; pq[1] += S[i].y * qr; pq[2] += S[i].z * qr; pq[3] += S[i].w * qr;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            s_red[0][rg][c0 + j] = pk[j];
            s_red[1][rg][c0 + j] = pq[j];
        }
        __syncthreads();
        if (tid < kSD) {
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int g = 0; g < kRowGroups; ++g) {
                sk += s_red[0][g][tid];
                sq += s_red[1][g][tid];
            }
            const float d = bt * (s_d[tid] - a * sk);
            s_d[tid] = d;
            static_cast<T*>(p.out)[(size_t)bh * kSD + tid] = from_f32<T>(p.scale * (a * sq + d * s_kq));
        }
        __syncthreads();
        const float d0 = s_d[c0 + 0], d1 = s_d[c0 + 1], d2 = s_d[c0 + 2], d3 = s_d[c0 + 3];
        float* Sp = p.state + (size_t)bh * kSD * kSD;
#pragma unroll
        for (int i = 0; i < kMaxRowsPerThread; ++i) {
            const int r = rg + i * kRowGroups;
            const float kr = s_k[r];
            float4 x;
            x.x = a * S[i].x + kr * d0;
            x.y = a * S[i].y + kr * d1;
            x.z = a * S[i].z + kr * d2;
            x.w = a * S[i].w + kr * d3;
            __stcs(reinterpret_cast<float4*>(Sp + (size_t)r * kSD + c0), x);
        }
    }
    __syncthreads();
    if (tid == 0 && sm.abort && status) atomicExch(status, (int32_t)GDN_ERR_TIMEOUT);
}

template <typename T>
cudaError_t launch_stream(const Problem& p, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(gdn_decode_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)sizeof(DecodeStreamSmem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int32_t* status = nullptr;
    if (status_word_for_current_device(&status) != GDN_OK) status = nullptr;
    const int heads = p.B * p.Hv;
    gdn_decode_stream_kernel<T><<<heads < 2 * sms ? heads : 2 * sms, kSThreads, sizeof(DecodeStreamSmem), stream>>>(
        p, status);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const Problem& p, cudaStream_t stream) {
    if (p.Dk == kSD && p.Dv == kSD) return launch_stream<T>(p, stream);
    dim3 grid(p.B * p.Hv, (p.Dv + kCols - 1) / kCols);
    const bool vec = (p.Dv % 4) == 0;
    const T* q = static_cast<const T*>(p.q);
    const T* k = static_cast<const T*>(p.k);
    const T* v = static_cast<const T*>(p.v);
    T* out = static_cast<T*>(p.out);
    if (vec)
        gdn_decode_kernel<T, true><<<grid, kThreads, 0, stream>>>(q, k, v, p.g_log, p.beta, p.scale, p.state, out,
                                                                  p.Hk, p.Hv, p.Dk, p.Dv, p.zero_init ? 1 : 0);
    else
        gdn_decode_kernel<T, false><<<grid, kThreads, 0, stream>>>(q, k, v, p.g_log, p.beta, p.scale, p.state,
                                                                   out, p.Hk, p.Hv, p.Dk, p.Dv,
                                                                   p.zero_init ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const Problem& p, cudaStream_t stream) {
    return p.bf16 ? launch_typed<__nv_bfloat16>(p, stream) : launch_typed<float>(p, stream);
}

}  // namespace gdn
