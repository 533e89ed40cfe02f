// decode_gated.cu -- the gated single-token step of the decode block: the
// decode prologue (L2-normalised q and k, the decay g and update strength beta
// from the raw gate inputs), one token of the recurrence, and the RMSNormGated
// output epilogue ("GDN Block TKG Kernel API Reference": gdn_block_tkg
// Parameters A_log, dt_bias, norm_weight and the z / a / b projections,
// Returns "RMSNormGated decode output"; the data flow into gdn_tkg).
//
//     q^ = q / sqrt(|q|^2 + eps_l2),  k^ likewise
//     g  = -exp(A_log[h]) softplus(a + dt_bias[h]),   beta = sigmoid(b)
//     p_k = S^T k^,  p_q = S^T q^,  d = beta (v - e^g p_k)
//     o  = scale (e^g p_q + d (k^ . q^)),   S' = e^g S + k^ d^T   (in place)
//     y  = o / sqrt(mean_Dv(o^2) + eps_rms) * norm_weight * silu(z)
//
// A CTA of 256 threads covers all Dv <= 128 columns of a head, because the RMS
// norm runs over the whole head: 32 column groups of 4 floats x 8 row groups.
// Every fp32 state element is read once and written once.  At Dk = Dv = 128
// with 16-byte aligned rows, persistent CTAs (two per SM) stream the heads
// through shared memory (gdn_decode_gated_stream_kernel); other shapes run one
// CTA per head (gdn_decode_gated_kernel).  Both share the per-head math
// (gated_head).  In its conv mode (the decode block) the kernel computes q, k, v
// from the shifted conv windows instead of reading them.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gdn_internal.h"
#include "gdn_device.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kColGroups = 32;  // x 4 columns = 128
constexpr int kRowGroups = 8;
constexpr int kMaxRows = 128 / kRowGroups;
constexpr float kEpsL2 = 1e-6f;
constexpr float kEpsRms = 1e-6f;


__device__ __forceinline__ float softplus(float x) { return x > 20.f ? x : log1pf(expf(x)); }

struct GatedArgs {
    const void* qkv;
    const void* z;
    const void* a;
    const void* b;
    const float* A_log;
    const float* dt_bias;
    const float* norm_weight;
    float scale;
    float* state;
    void* out;
    int Hk, Hv, Dk, Dv, zero_init;
    // conv mode: q|k|v come from the shifted conv windows [B, conv_dim, K] (bf16) and the
    // taps [conv_dim, K] fp32, conv_out = silu(sum_k w[c, k] window[b, c, k]) rounded to bf16
    const void* conv_win;
    const float* conv_w;
    int K;
    int32_t* status;  // device status word: a wait that gave up records GDN_ERR_TIMEOUT
    // Streaming kernel: when set, heads after each CTA's first are taken from this counter
    // (zero when the kernel starts reading it; advanced by one per head taken), so that CTAs
    // that start early take more heads.  When null, CTA i takes heads i, i + gridDim.x, ...
    int* next_head;
};

// How the kernel gets q, k and v: kDirect reads them; kConv4 / kConvAny compute the
// conv1d decode output from the window (K == 4 as one 8-byte word / any K).
enum InputMode { kDirect = 0, kConv4 = 1, kConvAny = 2 };


// conv1d decode output of one channel from its shifted window (4 bf16, oldest first, in one
// 8-byte word) and its taps, rounded to bf16 as the stand-alone conv step stores it
__device__ __forceinline__ float conv4_value(uint2 s, float4 w) {
    float z = fmaf(w.x, __uint_as_float(s.x << 16), 0.f);
    z = fmaf(w.y, __uint_as_float(s.x & 0xffff0000u), z);
    z = fmaf(w.z, __uint_as_float(s.y << 16), z);
    z = fmaf(w.w, __uint_as_float(s.y & 0xffff0000u), z);
    return __bfloat162float(__float2bfloat16_rn(silu_fast(z)));
}

template <typename T, int kMode>
__device__ __forceinline__ float input_value(const GatedArgs& p, const T* row_in, long long row, long long ch) {
    if constexpr (kMode == kDirect) {
        return to_f32(row_in[ch]);
    } else if constexpr (kMode == kConv4) {
        return conv4_value(reinterpret_cast<const uint2*>(p.conv_win)[row + ch],
                           reinterpret_cast<const float4*>(p.conv_w)[ch]);
    } else {
        const __nv_bfloat16* s = static_cast<const __nv_bfloat16*>(p.conv_win) + (row + ch) * p.K;
        const float* w = p.conv_w + ch * p.K;
        float z = 0.f;
        for (int k = 0; k < p.K; ++k) z = fmaf(w[k], __bfloat162float(s[k]), z);
        return __bfloat162float(__float2bfloat16_rn(silu_fast(z)));
    }
}

// Per-head scratch of the step (shared memory).
struct GatedShared {
    float s_k[128], s_q[128];  // raw q and k; their norms are applied to the reductions
    float s_red[2][kRowGroups][128];
    float s_d[128];
    float s_v[128], s_gate[128];  // v, and norm_weight * silu(z)
    float s_part[4][kThreads / 32];  // per-warp partial sums: |q|^2, |k|^2, k.q, sum o^2
};

// One head once its inputs are at hand: the state in registers (thread (rg, cg) holds rows
// rg + 8 i, columns 4 cg .. 4 cg + 3), raw q and k in registers (thread < Dk), v and
// norm_weight * silu(z) in sh.s_v / sh.s_gate (thread < Dv, written before the call), the raw
// gate inputs.  Computes the step, stores the new state in place and the gated output.
template <typename T, bool kVec>
__device__ __forceinline__ void gated_head(const GatedArgs& p, GatedShared& sh, int bh, float4 (&S)[kMaxRows],
                                           float qv, float kv, float a_in, float b_in, float A_log, float dt_bias) {
    float* s_k = sh.s_k;
    float* s_q = sh.s_q;
    auto& s_red = sh.s_red;
    float* s_d = sh.s_d;
    float* s_v = sh.s_v;
    float* s_gate = sh.s_gate;
    auto& s_part = sh.s_part;
    const int Dk = p.Dk, Dv = p.Dv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid & (kColGroups - 1), rg = tid >> 5;
    const int c0 = cg * 4;
    float* Sp = p.state + (long long)bh * Dk * Dv;

    if (tid < Dk) {
        s_q[tid] = qv;
        s_k[tid] = kv;
    }
    {
        const float sq = warp_sum(qv * qv), sk = warp_sum(kv * kv), skq = warp_sum(qv * kv);
        if (lane == 0) {
            s_part[0][warp] = sq;
            s_part[1][warp] = sk;
            s_part[2][warp] = skq;
        }
    }
    const float g = -expf(A_log) * softplus(a_in + dt_bias);
    const float decay = expf(g);
    const float beta = 1.f / (1.f + expf(-b_in));
    __syncthreads();
    float nq = 0.f, nk = 0.f, nkq = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        nq += s_part[0][w];
        nk += s_part[1][w];
        nkq += s_part[2][w];
    }
    const float inv_q = rsqrtf(nq + kEpsL2), inv_k = rsqrtf(nk + kEpsL2);
    const float kq = nkq * inv_q * inv_k;

    // S^T k and S^T q with the raw vectors: partials over this thread's rows, then over the row groups
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) {
        const int r = rg + i * kRowGroups;
        if (r < Dk) {
            const float kr = s_k[r], qr = s_q[r];
            pk[0] = fmaf(S[i].x, kr, pk[0]);
            pk[1] = fmaf(S[i].y, kr, pk[1]);
            pk[2] = fmaf(S[i].z, kr, pk[2]);
            pk[3] = fmaf(S[i].w, kr, pk[3]);
            pq[0] = fmaf(S[i].x, qr, pq[0]);
            pq[1] = fmaf(S[i].y, qr, pq[1]);
            pq[2] = fmaf(S[i].z, qr, pq[2]);
            pq[3] = fmaf(S[i].w, qr, pq[3]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s_red[0][rg][c0 + j] = pk[j];
        s_red[1][rg][c0 + j] = pq[j];
    }
    __syncthreads();
    float o = 0.f;
    if (tid < Dv) {
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int gi = 0; gi < kRowGroups; ++gi) {
            sk += s_red[0][gi][tid];
            sq += s_red[1][gi][tid];
        }
        const float d = beta * (s_v[tid] - decay * (sk * inv_k));
        s_d[tid] = d;
        o = p.scale * (decay * (sq * inv_q) + d * kq);
    }
    {
        const float so = warp_sum(o * o);
        if (lane == 0) s_part[3][warp] = so;
    }
    __syncthreads();

    // S' = e^g S + k^ d^T, in place; the stores go out before the output epilogue
    const float d0 = s_d[c0 + 0], d1 = s_d[c0 + 1], d2 = s_d[c0 + 2], d3 = s_d[c0 + 3];
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) {
        const int r = rg + i * kRowGroups;
        if (r < Dk) {
            const float kr = s_k[r] * inv_k;
            float4 x;
            x.x = fmaf(decay, S[i].x, kr * d0);
            x.y = fmaf(decay, S[i].y, kr * d1);
            x.z = fmaf(decay, S[i].z, kr * d2);
            x.w = fmaf(decay, S[i].w, kr * d3);
            if (kVec) {
                if (c0 < Dv) __stcs(reinterpret_cast<float4*>(Sp + (long long)r * Dv + c0), x);
            } else {
                float* row = Sp + (long long)r * Dv;
                if (c0 + 0 < Dv) row[c0 + 0] = x.x;
                if (c0 + 1 < Dv) row[c0 + 1] = x.y;
                if (c0 + 2 < Dv) row[c0 + 2] = x.z;
                if (c0 + 3 < Dv) row[c0 + 3] = x.w;
            }
        }
    }

    // epilogue: RMS of o over the head, gate, store
    if (tid < Dv) {
        float so = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) so += s_part[3][w];
        const float rinv = rsqrtf(so / (float)Dv + kEpsRms);
        static_cast<T*>(p.out)[(long long)bh * Dv + tid] = from_f32<T>(o * rinv * s_gate[tid]);
    }
}


template <typename T, bool kVec, int kMode>
__global__ void __launch_bounds__(kThreads, 2) gdn_decode_gated_kernel(GatedArgs p) {
    __shared__ GatedShared sh;
    const int bh = blockIdx.x;
    const int Hv = p.Hv, Dk = p.Dk, Dv = p.Dv;
    const int b = bh / Hv, h = bh - b * Hv;
    const int hk = h / (Hv / p.Hk);
    const int tid = threadIdx.x;
    const int cg = tid & (kColGroups - 1), rg = tid >> 5;
    const int c0 = cg * 4;
    const long long conv_dim = 2LL * p.Hk * Dk + (long long)Hv * Dv;
    const T* row_in = static_cast<const T*>(p.qkv) + b * conv_dim;  // kDirect
    const long long row = (long long)b * conv_dim;                     // conv modes
    const long long ch_q = (long long)hk * Dk, ch_k = (long long)p.Hk * Dk + ch_q;
    const long long ch_v = 2LL * p.Hk * Dk + (long long)h * Dv;
    const float* Sp = p.state + (long long)bh * Dk * Dv;

    // the state loads go out first: they are the bulk of the traffic
    float4 S[kMaxRows];
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) {
        const int r = rg + i * kRowGroups;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!p.zero_init && r < Dk) {
            if (kVec) {
                if (c0 < Dv) x = __ldcs(reinterpret_cast<const float4*>(Sp + (long long)r * Dv + c0));
            } else {
                const float* rowp = Sp + (long long)r * Dv;
                if (c0 + 0 < Dv) x.x = rowp[c0 + 0];
                if (c0 + 1 < Dv) x.y = rowp[c0 + 1];
                if (c0 + 2 < Dv) x.z = rowp[c0 + 2];
                if (c0 + 3 < Dv) x.w = rowp[c0 + 3];
            }
        }
        S[i] = x;
    }
    // Behind a programmatic launch the loads above overlap the producer of the
    // inputs below (the decode block's projection kernel); the state is not its output.
    ptx::griddep_wait();

    // every other input of the head is fetched now too, so that no load waits behind a barrier
    float qv = 0.f, kv = 0.f;
    if (tid < Dk) {
        qv = input_value<T, kMode>(p, row_in, row, ch_q + tid);
        kv = input_value<T, kMode>(p, row_in, row, ch_k + tid);
    }
    if (tid < Dv) {
        const float zv = to_f32(static_cast<const T*>(p.z)[(long long)bh * Dv + tid]);
        sh.s_v[tid] = input_value<T, kMode>(p, row_in, row, ch_v + tid);
        sh.s_gate[tid] = p.norm_weight[tid] * (zv / (1.f + expf(-zv)));
    }
    const float a_in = to_f32(static_cast<const T*>(p.a)[bh]), b_in = to_f32(static_cast<const T*>(p.b)[bh]);
    gated_head<T, kVec>(p, sh, bh, S, qv, kv, a_in, b_in, p.A_log[h], p.dt_bias[h]);
}

// Dk = Dv = 128 with 16-byte aligned state and input rows: persistent CTAs, two per SM,
// walk the heads blockIdx.x, blockIdx.x + gridDim.x, ...  A head's state (64 KB) reaches
// shared memory in one bulk copy and its other inputs in 16-byte asynchronous copies, both
// issued as soon as the previous head has been read out of shared memory, so that the
// memory system holds the next head's bytes while the CTA computes.  The step itself is
// gated_head, as in gdn_decode_gated_kernel.
constexpr int kSD = 128;
constexpr uint32_t kStreamStateBytes = kSD * kSD * 4;
constexpr uint32_t kStreamInBytes = 9984;  // the largest input set (conv mode, below)

struct StreamSmem {
    float state[kSD * kSD];
    alignas(16) uint8_t in[kStreamInBytes];
    uint64_t full;
    int abort;
};

// Input buffer of one head.  Direct: q, k, v, z [128] in the compute type at 0, 128, 256,
// 384 elements, then norm_weight [128] fp32.  Conv mode: the windows of the q, k, v channels
// [128] uint2 at bytes 0, 1024, 2048, their taps [128] float4 at 3072, 5120, 7168, z [128]
// bf16 at 9216, norm_weight [128] fp32 at 9472.
template <typename T, int kMode>
__device__ __forceinline__ void stream_issue_inputs(const GatedArgs& p, uint8_t* in, int bh) {
    const int Hv = p.Hv, b = bh / Hv, h = bh - b * Hv, hk = h / (Hv / p.Hk);
    const long long C = 2LL * p.Hk * kSD + (long long)Hv * kSD;
    const long long cq = (long long)hk * kSD, ck = (long long)p.Hk * kSD + cq, cv = 2LL * p.Hk * kSD + (long long)h * kSD;
    const uint8_t* src[8];
    uint32_t off[8], bytes[8];
    int n = 0;
    auto add = [&](const void* sp, uint32_t o, uint32_t nb) {
        src[n] = static_cast<const uint8_t*>(sp);
        off[n] = o;
        bytes[n] = nb;
        ++n;
    };
    if constexpr (kMode == kDirect) {
        constexpr uint32_t e = sizeof(T);
        const T* rowp = static_cast<const T*>(p.qkv) + (long long)b * C;
        add(rowp + cq, 0, kSD * e);
        add(rowp + ck, kSD * e, kSD * e);
        add(rowp + cv, 2 * kSD * e, kSD * e);
        add(static_cast<const T*>(p.z) + (long long)bh * kSD, 3 * kSD * e, kSD * e);
        add(p.norm_weight, 4 * kSD * e, kSD * 4);
    } else {
        const uint2* win = static_cast<const uint2*>(p.conv_win) + (long long)b * C;
        const float4* taps = reinterpret_cast<const float4*>(p.conv_w);
        add(win + cq, 0, 1024);
        add(win + ck, 1024, 1024);
        add(win + cv, 2048, 1024);
        add(taps + cq, 3072, 2048);
        add(taps + ck, 5120, 2048);
        add(taps + cv, 7168, 2048);
        add(static_cast<const __nv_bfloat16*>(p.z) + (long long)bh * kSD, 9216, 256);
        add(p.norm_weight, 9472, 512);
    }
    for (int r = 0; r < n; ++r)
        for (uint32_t i = threadIdx.x; i < bytes[r] / 16; i += kThreads) ptx::cp_async_16(in + off[r] + 16 * i, src[r] + 16 * i);
    ptx::cp_async_commit();
}

template <typename T, int kMode>
__global__ void __launch_bounds__(kThreads, 2) gdn_decode_gated_stream_kernel(GatedArgs p, int num_heads) {
    extern __shared__ __align__(128) uint8_t stream_raw[];
    StreamSmem& sm = *reinterpret_cast<StreamSmem*>(stream_raw);
    __shared__ GatedShared sh;
    const int tid = threadIdx.x;
    const int cg = tid & (kColGroups - 1), rg = tid >> 5, c0 = cg * 4;
    auto load_state = [&](int bh) {
        ptx::mbar_arrive_expect_tx(&sm.full, kStreamStateBytes);
        ptx::bulk_load_evict_first(sm.state, p.state + (long long)bh * kSD * kSD, kStreamStateBytes, &sm.full);
    };
    __shared__ int s_next;
    if (tid == 0) {
        ptx::mbar_init(&sm.full, 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    int bh = (int)blockIdx.x;  // the CTA's first head (the grid has at most num_heads CTAs)
    if (tid == 0 && !p.zero_init) load_state(bh);
    // Behind a programmatic launch the state copy above overlaps the producer of the other
    // inputs (the decode block's projection kernel); the state is not its output.
    ptx::griddep_wait();
    stream_issue_inputs<T, kMode>(p, sm.in, bh);
    float a_n = to_f32(static_cast<const T*>(p.a)[bh]), b_n = to_f32(static_cast<const T*>(p.b)[bh]);
    float al_n = p.A_log[bh % p.Hv], dt_n = p.dt_bias[bh % p.Hv];

    for (int l = 0;; ++l) {
        const float a_in = a_n, b_in = b_n, A_log = al_n, dt_bias = dt_n;
        if (!p.zero_init) (void)ptx::mbar_wait_or_abort(&sm.full, l & 1, &sm.abort);
        ptx::cp_async_wait_all();
        __syncthreads();  // every thread's copies have landed; the previous head is done with sh
        float4 S[kMaxRows];
#pragma unroll
        for (int i = 0; i < kMaxRows; ++i)
            S[i] = p.zero_init ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : *reinterpret_cast<const float4*>(&sm.state[(rg + i * kRowGroups) * kSD + c0]);
        float qv = 0.f, kv = 0.f, vv = 0.f, zv = 0.f, nw = 0.f;
        if (tid < kSD) {
            if constexpr (kMode == kDirect) {
                const T* in = reinterpret_cast<const T*>(sm.in);
                qv = to_f32(in[tid]);
                kv = to_f32(in[kSD + tid]);
                vv = to_f32(in[2 * kSD + tid]);
                zv = to_f32(in[3 * kSD + tid]);
                nw = reinterpret_cast<const float*>(sm.in + 4 * kSD * sizeof(T))[tid];
            } else {
                const uint2* win = reinterpret_cast<const uint2*>(sm.in);
                const float4* taps = reinterpret_cast<const float4*>(sm.in + 3072);
                qv = conv4_value(win[tid], taps[tid]);
                kv = conv4_value(win[kSD + tid], taps[kSD + tid]);
                vv = conv4_value(win[2 * kSD + tid], taps[2 * kSD + tid]);
                zv = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(sm.in + 9216)[tid]);
                nw = reinterpret_cast<const float*>(sm.in + 9472)[tid];
            }
        }
        if (tid == 0) s_next = p.next_head ? atomicAdd(p.next_head, 1) + (int)gridDim.x : bh + (int)gridDim.x;
        __syncthreads();  // the state and the inputs of this head have been read out of shared memory
        const int nb = s_next;
        if (nb < num_heads) {
            if (tid == 0 && !p.zero_init) load_state(nb);
            stream_issue_inputs<T, kMode>(p, sm.in, nb);
            a_n = to_f32(static_cast<const T*>(p.a)[nb]);
            b_n = to_f32(static_cast<const T*>(p.b)[nb]);
            al_n = p.A_log[nb % p.Hv];
            dt_n = p.dt_bias[nb % p.Hv];
        }
        if (tid < kSD) {
            sh.s_v[tid] = vv;
            sh.s_gate[tid] = nw * (zv / (1.f + expf(-zv)));
        }
        gated_head<T, true>(p, sh, bh, S, qv, kv, a_in, b_in, A_log, dt_bias);
        if (nb >= num_heads) break;
        bh = nb;
    }
    __syncthreads();
    if (tid == 0 && sm.abort) atomicExch(p.status, (int32_t)GDN_ERR_TIMEOUT);
}

template <typename T, int kMode>
cudaError_t launch_stream(const GatedArgs& a, int B, cudaStream_t s, bool after_producer) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(gdn_decode_gated_stream_kernel<T, kMode>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(StreamSmem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int heads = B * a.Hv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(heads < 2 * sms ? heads : 2 * sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(StreamSmem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_producer ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gdn_decode_gated_stream_kernel<T, kMode>, a, heads);
}

// The streaming kernel needs Dk = Dv = 128 and 16-byte aligned state, input rows and taps.
bool stream_ok(const GatedArgs& a, size_t esz) {
    const auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    const long long C = 2LL * a.Hk * a.Dk + (long long)a.Hv * a.Dv;
    if (a.Dk != kSD || a.Dv != kSD || !al(a.state) || !al(a.z) || !al(a.norm_weight)) return false;
    if (a.conv_win) return a.K == 4 && al(a.conv_win) && al(a.conv_w);
    return al(a.qkv) && (C * (long long)esz) % 16 == 0;
}

template <typename T, bool kVec, int kMode>
cudaError_t launch_one(const GatedArgs& a, int B, cudaStream_t s, bool after_producer) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * a.Hv));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_producer ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gdn_decode_gated_kernel<T, kVec, kMode>, a);
}

template <typename T>
cudaError_t launch_gated(const GatedArgs& a, int B, cudaStream_t s, bool after_producer) {
    if (stream_ok(a, sizeof(T))) return launch_stream<T, kDirect>(a, B, s, after_producer);
    const bool vec = (a.Dv % 4) == 0 && (reinterpret_cast<uintptr_t>(a.state) & 15u) == 0;
    return vec ? launch_one<T, true, kDirect>(a, B, s, after_producer)
               : launch_one<T, false, kDirect>(a, B, s, after_producer);
}

cudaError_t launch_gated_conv(const GatedArgs& a, int B, cudaStream_t s, bool after_producer) {
    using T = __nv_bfloat16;
    const bool vec = (a.Dv % 4) == 0 && (reinterpret_cast<uintptr_t>(a.state) & 15u) == 0;
    const bool conv4 = a.K == 4 && (reinterpret_cast<uintptr_t>(a.conv_win) & 7u) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.conv_w) & 15u) == 0;
    if (conv4 && stream_ok(a, sizeof(T))) return launch_stream<T, kConv4>(a, B, s, after_producer);
    if (conv4)
        return vec ? launch_one<T, true, kConv4>(a, B, s, after_producer)
                   : launch_one<T, false, kConv4>(a, B, s, after_producer);
    return vec ? launch_one<T, true, kConvAny>(a, B, s, after_producer)
               : launch_one<T, false, kConvAny>(a, B, s, after_producer);
}

}  // namespace
}  // namespace gdn

gdn_status gdn::decode_gated_checked(const void* qkv, const void* z, const void* a, const void* b,
                                     const float* A_log, const float* dt_bias, const float* norm_weight, float scale,
                                     float* state_inout, void* out, const gdn_dims* d, cudaStream_t s,
                                     bool after_producer, const GatedConvInput* conv, int* next_head) {
    if (!d) return GDN_ERR_NULL;
    if (d->dtype != GDN_F32 && d->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (d->flags & ~(uint32_t)GDN_ZERO_INITIAL_STATE) return GDN_ERR_UNSUPPORTED;
    if (d->B < 0 || d->Hk < 1 || d->Hv < 1 || d->S != 1 || d->Dk < 1 || d->Dv < 1) return GDN_ERR_DIMS;
    if (d->Dk > 128 || d->Dv > 128 || d->Hv % d->Hk != 0) return GDN_ERR_DIMS;
    if (d->B * d->Hv > INT32_MAX) return GDN_ERR_DIMS;
    if (d->B == 0) return GDN_OK;
    if (conv && (d->dtype != GDN_BF16 || !conv->window || !conv->weight || conv->K < 1)) return GDN_ERR_UNSUPPORTED;
    if ((!qkv && !conv) || !z || !a || !b || !A_log || !dt_bias || !norm_weight || !state_inout || !out) return GDN_ERR_NULL;
    const uintptr_t esz = d->dtype == GDN_BF16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(a) |
         reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(out)) & (esz - 1))
        return GDN_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(A_log) | reinterpret_cast<uintptr_t>(dt_bias) |
         reinterpret_cast<uintptr_t>(norm_weight) | reinterpret_cast<uintptr_t>(state_inout)) & 3u)
        return GDN_ERR_ALIGN;
    GatedArgs g{qkv, z, a, b, A_log, dt_bias, norm_weight, scale, state_inout, out,
                (int)d->Hk, (int)d->Hv, (int)d->Dk, (int)d->Dv, (d->flags & GDN_ZERO_INITIAL_STATE) ? 1 : 0,
                conv ? conv->window : nullptr, conv ? conv->weight : nullptr, conv ? conv->K : 0, nullptr, next_head};
    gdn_status sw = status_word_for_current_device(&g.status);
    if (sw != GDN_OK) return sw;
    const cudaError_t e = conv ? launch_gated_conv(g, (int)d->B, s, after_producer)
                          : d->dtype == GDN_BF16 ? launch_gated<__nv_bfloat16>(g, (int)d->B, s, after_producer)
                                                 : launch_gated<float>(g, (int)d->B, s, after_producer);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_decode_gated(const void* qkv, const void* z, const void* a, const void* b,
                                       const float* A_log, const float* dt_bias, const float* norm_weight,
                                       float scale, float* state_inout, void* out, const gdn_dims* d,
                                       gdn_stream_t stream) {
    return gdn::decode_gated_checked(qkv, z, a, b, A_log, dt_bias, norm_weight, scale, state_inout, out, d,
                                     reinterpret_cast<cudaStream_t>(stream), false, nullptr, nullptr);
}
