// block.cu -- the decode block without its output projection ("GDN Block TKG
// Kernel API Reference": gdn_block_tkg Parameters, Returns, Notes and the data
// flow "in_proj matmuls -> gdn_conv1d_decode -> split conv_out + GQA-repeat q,k
// -> gdn_tkg").  Two launches on the caller's stream:
//
//   1. the four input projections of the token's hidden state, one grouped
//      tcgen05 GEMM (this file): [B, H] x [H, N] for N = conv_dim, value_dim,
//      num_v_heads, num_v_heads.  z, a and b go to the caller's workspace in
//      bf16.  The q|k|v projection is not written out: the thread that holds
//      its output column n holds channel n for every token, so it shifts that
//      channel's conv window in place, appending the new value (rounded to
//      bf16) -- the window then holds everything the conv1d decode step needs;
//   2. the gated step (decode_gated.cu) in its conv mode: each q, k, v value is
//      silu(sum_k w[c, k] window[b, c, k]), rounded to bf16, computed where it
//      is consumed -- the arithmetic, tap order and roundings of
//      gdn_conv1d_decode.  It is launched as a programmatic dependent of the
//      GEMM: its CTAs start once every GEMM CTA is resident, load their fp32
//      state while the GEMM runs, and wait for it before reading its outputs.
//
// The GEMM is a weight stream (M = B tokens is small): each CTA owns 128 output
// columns of one weight matrix and runs over H in 64-row slabs.  The product is
// issued transposed, D^T[n][b] = sum_h W[h][n] X[b][h], so the 128 columns sit on
// the tcgen05 M / TMEM-lane axis and the batch on N: A = the W slab (MN-major,
// two 64-column boxes with the 128-byte swizzle), B = the hidden rows (K-major).
// Warp 0 issues the TMA loads through args.stages stages, warp 1 the MMAs, warps
// 2..5 write the fp32 accumulator back as bf16 (one TMEM lane quadrant each).
// While the main loop runs, the epilogue warps of the q|k|v CTAs copy their conv
// windows (B <= 64) to shared memory with cp.async.  The pipeline is as deep as
// 200 KB of shared memory allows, which leaves room for a CTA of the gated step.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "gdn_internal.h"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kGTile = 128;   // output columns per CTA
constexpr int kSlab = 64;     // hidden rows per stage
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;   // leaves room for a CTA of the gated step on the same SM
constexpr int kWinTokens = 64;            // conv windows staged in shared memory up to this batch
constexpr int kGThreads = 192;
constexpr uint32_t kBoxBytes = 64 * 128;  // [64 rows][64 bf16]
constexpr int kMaxGroups = 4;

struct GemmArgs {
    void* out[kMaxGroups];        // [B][N_g] bf16 (group 0: none, its values go to the windows)
    int N[kMaxGroups];
    __nv_bfloat16* conv_state;    // [B][N_0][K]: group 0's conv windows, shifted in place
    int K, conv_vec4;             // conv_vec4: K == 4 with 8-byte windows
    int* head_counter;            // the gated step's head counter, zeroed here
    int tile_start[kMaxGroups + 1];
    int B, H, nb, npad;           // nb = hidden boxes of 64 rows; npad = MMA N
    int stages;                   // pipeline depth, <= kMaxStages
    uint32_t stage_bytes, tmem_cols, idesc;
    uint32_t win_off, win_bytes;  // staged conv windows [B][kGTile] uint2 (0 bytes: read from global)
    int32_t* status;
};

struct GemmBars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

__global__ void __launch_bounds__(kGThreads, 2)
    inproj_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w0,
                       const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_w2,
                       const __grid_constant__ CUtensorMap tm_w3, const __grid_constant__ GemmArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    const int stages = args.stages;
    GemmBars* bars = reinterpret_cast<GemmBars*>(sm + stages * args.stage_bytes);
    volatile int* abort_flag = &bars->abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    ptx::griddep_launch_dependents();  // the gated step may start its state loads now
    if (blockIdx.x == 0 && tid == 0) *args.head_counter = 0;  // read by the gated step after this grid completes

    int g = 0;  // weight matrix of this CTA
    while (g + 1 < kMaxGroups && (int)blockIdx.x >= args.tile_start[g + 1]) ++g;
    const int n0 = ((int)blockIdx.x - args.tile_start[g]) * kGTile;
    const CUtensorMap* tm_w = g == 0 ? &tm_w0 : g == 1 ? &tm_w1 : g == 2 ? &tm_w2 : &tm_w3;
    const int n_slabs = args.H / kSlab;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->done, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, args.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // TMA producer
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(tm_w);
            int loaded = 0;
            for (int i = 0; i < n_slabs; ++i) {
                const int s = i % stages;
                if (i >= stages && !mbar_wait_or_abort(&bars->empty[s], ((i / stages) - 1) & 1, abort_flag)) break;
                uint8_t* st = sm + s * args.stage_bytes;
                mbar_arrive_expect_tx(&bars->full[s], args.stage_bytes);
                tma_load_3d(st, tm_w, &bars->full[s], n0, i * kSlab, 0);
                tma_load_3d(st + kBoxBytes, tm_w, &bars->full[s], n0 + 64, i * kSlab, 0);
                for (int j = 0; j < args.nb; ++j)
                    tma_load_3d(st + 2 * kBoxBytes + j * kBoxBytes, &tm_x, &bars->full[s], i * kSlab, j * 64, 0);
                loaded = i + 1;
            }
            // drain: every issued load has landed before the CTA can exit (bounded)
            for (int i = (loaded > stages ? loaded - stages : 0); i < loaded; ++i)
                (void)mbar_wait(&bars->full[i % stages], (i / stages) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            int issued = 0;
            for (int i = 0; i < n_slabs; ++i) {
                const int s = i % stages;
                if (!mbar_wait_or_abort(&bars->full[s], (i / stages) & 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t st = sbase + s * args.stage_bytes;
                const uint64_t dw = make_sdesc(st, kBoxBytes, 1024), dx = make_sdesc(st + 2 * kBoxBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kSlab / 16; ++kk)
                    mma_bf16(tmem, sdesc_add(dw, kk * 2048), sdesc_add(dx, kk * 32), args.idesc, (i > 0 || kk > 0));
                mma_commit(&bars->empty[s]);
                issued = i + 1;
            }
            if (issued == n_slabs) {
                mma_commit(&bars->done);
            } else if (issued > 0) {  // drain what was issued (bounded)
                (void)mbar_wait(&bars->empty[(issued - 1) % stages], ((issued - 1) / stages) & 1);
            }
        }
    } else {  // epilogue: warps 2..5 cover the four lane quadrants
        const int quad = warp & 3;
        const int n = n0 + quad * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        const int N = args.N[g];
        const bool conv = g == 0;
        // while the main loop runs, this thread's conv windows (channel n, every token) are
        // copied to shared memory, so that the epilogue does not wait on them
        uint2* win = reinterpret_cast<uint2*>(sm + args.win_off) + quad * 32 + lane;
        const bool staged = conv && args.win_bytes != 0 && n < N;
        if (staged) {
            const uint2* src = reinterpret_cast<const uint2*>(args.conv_state) + n;
            for (int b = 0; b < args.B; ++b) cp_async_8(win + b * kGTile, src + (size_t)b * N);
            cp_async_commit();
        }
        const bool ok = mbar_wait_or_abort(&bars->done, 0, abort_flag);
        tc_fence_after();
        if (staged) cp_async_wait_all();
        if (ok) {
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out[g]);
#pragma unroll 1
            for (int b0 = 0; b0 < args.npad; b0 += 32) {
                float x[32];
                tmem_ld32(trow + b0, x);
                tmem_wait_ld();
                if (n >= N) continue;
                if (!conv) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (b0 + j < args.B) out[(size_t)(b0 + j) * N + n] = __float2bfloat16_rn(x[j]);
                } else if (args.conv_vec4) {
                    // window = 4 bf16 (oldest first) in one 8-byte word: drop the oldest, append x
                    uint2* sp = reinterpret_cast<uint2*>(args.conv_state) + (size_t)b0 * N + n;
#pragma unroll
                    for (int h = 0; h < 32; h += 16) {
                        uint2 sv[16];
                        if (staged) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                sv[j] = (b0 + h + j < args.B) ? win[(b0 + h + j) * kGTile] : make_uint2(0u, 0u);
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                sv[j] = (b0 + h + j < args.B) ? sp[(size_t)(h + j) * N] : make_uint2(0u, 0u);
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            if (b0 + h + j >= args.B) continue;
                            const uint32_t xb = __bfloat16_as_ushort(__float2bfloat16_rn(x[h + j]));
                            sp[(size_t)(h + j) * N] =
                                make_uint2((sv[j].x >> 16) | (sv[j].y << 16), (sv[j].y >> 16) | (xb << 16));
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (b0 + j >= args.B) continue;
                        __nv_bfloat16* sp = args.conv_state + ((size_t)(b0 + j) * N + n) * args.K;
                        for (int k = 0; k + 1 < args.K; ++k) sp[k] = sp[k + 1];
                        sp[args.K - 1] = __float2bfloat16_rn(x[j]);
                    }
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && bars->abort) atomicExch(args.status, (int32_t)GDN_ERR_TIMEOUT);
    if (warp == 1) tmem_dealloc(tmem, args.tmem_cols);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A [rows][cols] bf16 matrix (cols contiguous) as a 3-D map with a unit last
// dimension, boxes of 64 x 64 with the 128-byte swizzle; out-of-range rows and
// columns of a box read as zero.
bool encode_2d(CUtensorMap* map, const void* ptr, long long rows, long long cols) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
    cuuint32_t box[3] = {64, 64, 1}, estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct BlockLayout {
    long long C, VD;           // conv_dim, value_dim
    size_t off_z, off_a, off_b, off_ctr, bytes;
};

BlockLayout layout(const gdn_block_dims* d) {
    BlockLayout L;
    L.C = 2 * d->Hk * d->Dk + d->Hv * d->Dv;
    L.VD = d->Hv * d->Dv;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    size_t o = 0;
    L.off_z = o;    o = up(o + (size_t)d->B * L.VD * 2);
    L.off_a = o;    o = up(o + (size_t)d->B * d->Hv * 2);
    L.off_b = o;    o = up(o + (size_t)d->B * d->Hv * 2);
    L.off_ctr = o;  o = up(o + sizeof(int));
    L.bytes = o;
    return L;
}

gdn_status check_block(const gdn_block_dims* d) {
    if (!d) return GDN_ERR_NULL;
    if (d->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;  // bf16 weights and activations (Parameters)
    if (d->flags != 0) return GDN_ERR_UNSUPPORTED;
    if (d->B < 0 || d->H < 1 || d->Hk < 1 || d->Hv < 1 || d->Dk < 1 || d->Dv < 1 || d->K < 1) return GDN_ERR_DIMS;
    if (d->Dk > 128 || d->Dv > 128 || d->Hv % d->Hk != 0) return GDN_ERR_DIMS;
    if (d->K > 8 || d->B > 256 || d->H % 64 != 0) return GDN_ERR_UNSUPPORTED;
    const long long C = 2 * d->Hk * d->Dk + d->Hv * d->Dv;
    // TMA row pitches are multiples of 16 bytes
    if (C % 8 != 0 || (d->Hv * d->Dv) % 8 != 0 || d->Hv % 8 != 0) return GDN_ERR_UNSUPPORTED;
    if (C > INT32_MAX || d->B * C > INT32_MAX) return GDN_ERR_DIMS;
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" size_t gdn_decode_block_workspace_bytes(const gdn_block_dims* dims) {
    if (check_block(dims) != GDN_OK) return 0;
    return layout(dims).bytes;
}

extern "C" gdn_status gdn_decode_block(const void* hidden, const void* W_qkv, const void* W_z, const void* W_a,
                                       const void* W_b, const float* conv_weight, void* conv_state_inout,
                                       const float* A_log, const float* dt_bias, const float* norm_weight,
                                       float* state_inout, void* out, void* workspace, size_t workspace_bytes,
                                       const gdn_block_dims* d, gdn_stream_t stream) {
    gdn_status st = check_block(d);
    if (st != GDN_OK || d->B == 0) return st;
    if (!hidden || !W_qkv || !W_z || !W_a || !W_b || !conv_weight || !conv_state_inout || !A_log || !dt_bias ||
        !norm_weight || !state_inout || !out || !workspace)
        return GDN_ERR_NULL;
    const void* aligned_ptrs[] = {hidden, W_qkv, W_z, W_a, W_b, workspace};
    for (const void* p : aligned_ptrs)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return GDN_ERR_ALIGN;
    // element alignment of the rest, checked before the first launch
    if ((reinterpret_cast<uintptr_t>(conv_state_inout) | reinterpret_cast<uintptr_t>(out)) & 1u) return GDN_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(conv_weight) | reinterpret_cast<uintptr_t>(A_log) |
         reinterpret_cast<uintptr_t>(dt_bias) | reinterpret_cast<uintptr_t>(norm_weight) |
         reinterpret_cast<uintptr_t>(state_inout)) & 3u)
        return GDN_ERR_ALIGN;
    const BlockLayout L = layout(d);
    if (workspace_bytes < L.bytes) return GDN_ERR_DIMS;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // 1. the four input projections
    CUtensorMap tx, tw[kMaxGroups];
    const void* W[kMaxGroups] = {W_qkv, W_z, W_a, W_b};
    const long long N[kMaxGroups] = {L.C, L.VD, d->Hv, d->Hv};
    void* outs[kMaxGroups] = {nullptr, ws + L.off_z, ws + L.off_a, ws + L.off_b};
    if (!encode_2d(&tx, hidden, d->B, d->H)) return GDN_ERR_CUDA;
    GemmArgs a{};
    int tiles = 0;
    for (int g = 0; g < kMaxGroups; ++g) {
        if (!encode_2d(&tw[g], W[g], d->H, N[g])) return GDN_ERR_CUDA;
        a.out[g] = outs[g];
        a.N[g] = (int)N[g];
        a.tile_start[g] = tiles;
        tiles += (int)((N[g] + kGTile - 1) / kGTile);
    }
    a.tile_start[kMaxGroups] = tiles;
    a.conv_state = static_cast<__nv_bfloat16*>(conv_state_inout);
    a.head_counter = reinterpret_cast<int*>(ws + L.off_ctr);
    a.K = (int)d->K;
    a.conv_vec4 = d->K == 4 && (reinterpret_cast<uintptr_t>(conv_state_inout) & 7u) == 0;
    a.B = (int)d->B;
    a.H = (int)d->H;
    a.nb = (int)((d->B + 63) / 64);
    a.npad = (int)((d->B + 15) / 16 * 16);
    a.stage_bytes = 2 * kBoxBytes + a.nb * kBoxBytes;
    a.win_bytes = (a.B <= kWinTokens && a.conv_vec4) ? (uint32_t)(a.B * kGTile * 8) : 0u;
    {
        const int fixed = (int)((sizeof(GemmBars) + 15) & ~(size_t)15) + (int)a.win_bytes + 1024;
        a.stages = (kSmemBudget - fixed) / (int)a.stage_bytes;
        if (a.stages > kMaxStages) a.stages = kMaxStages;
    }
    a.win_off = (uint32_t)(a.stages * a.stage_bytes + ((sizeof(GemmBars) + 15) & ~(size_t)15));
    uint32_t cols = 32;
    while (cols < (uint32_t)a.npad) cols <<= 1;
    a.tmem_cols = cols;
    a.idesc = make_idesc_bf16(128, a.npad, 1, 0);
    if ((st = status_word_for_current_device(&a.status)) != GDN_OK) return st;
    const size_t smem = a.win_off + a.win_bytes + 1024;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(inproj_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSmemBudget);
    });
    if (attr_err != cudaSuccess) return GDN_ERR_CUDA;
    inproj_gemm_kernel<<<tiles, kGThreads, smem, s>>>(tx, tw[0], tw[1], tw[2], tw[3], a);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;

    // 2. the conv output and the gated step, behind the GEMM
    const gdn_dims gd{d->B, d->Hk, d->Hv, 1, d->Dk, d->Dv, GDN_BF16, 0};
    const GatedConvInput conv{conv_state_inout, conv_weight, (int)d->K};
    return decode_gated_checked(nullptr, ws + L.off_z, ws + L.off_a, ws + L.off_b, A_log, dt_bias, norm_weight,
                                1.0f / std::sqrt((float)d->Dk), state_inout, out, &gd, s, true, &conv,
                                reinterpret_cast<int*>(ws + L.off_ctr));
}

// ------------------------------------------------------------------ fixed-scratch variant
// gdn_decode_block_noalloc: the same two launches, with the inter-stage scratch (z, a, b and
// the head counter) in a fixed array of this library instead of a caller's workspace, for
// callers that cannot allocate device memory themselves.  Each CUDA device that loads the
// library holds its own copy of the array until the process exits.  Host code may not use
// the array's name as a device address (on the host it names a stand-in object), so its
// device address is looked up once per device with cudaGetSymbolAddress while that device
// is current, and handed to the kernels like a workspace pointer.
static __device__ __align__(256) uint8_t g_block_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace gdn {
namespace {
constexpr int kScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kScratchDevices] = {};

// Device address of the current device's scratch array (looked up on the first call per device).
gdn_status block_scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_block_scratch) != cudaSuccess) {
            (void)cudaGetLastError();
            return GDN_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}
}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_decode_block_noalloc(const void* hidden, const void* W_qkv, const void* W_z, const void* W_a,
                                               const void* W_b, const float* conv_weight, void* conv_state_inout,
                                               const float* A_log, const float* dt_bias, const float* norm_weight,
                                               float* state_inout, void* out, const gdn_block_dims* d,
                                               gdn_stream_t stream) {
    gdn_status st = check_block(d);
    if (st != GDN_OK || d->B == 0) return st;
    // z, a, b and the counter must fit the fixed array; the GEMM overwrites z, a and b and
    // zeroes the counter on every call, so nothing left by an earlier call is read
    if (layout(d).bytes > GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_UNSUPPORTED;
    void* ws = nullptr;
    if ((st = block_scratch_for_current_device(&ws)) != GDN_OK) return st;
    return gdn_decode_block(hidden, W_qkv, W_z, W_a, W_b, conv_weight, conv_state_inout, A_log, dt_bias, norm_weight,
                            state_inout, out, ws, GDN_NOALLOC_SCRATCH_BYTES, d, stream);
}
